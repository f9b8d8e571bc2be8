// kernels.h -- internal launch interface between the C-ABI layer (api.cu) and
// the kernels.  Host-side argument checking happens in api.cu; these launchers
// assume valid arguments.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace i8kv {

struct ProducerParams {
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* slots;
  int T, Hkv, D, num_blocks;
  int8_t* k_cache;
  int8_t* v_cache;
  float* k_scale;
  float* v_scale;
  const uint16_t* q;  // nullable
  int Hq;
  int8_t* q_i8;  // nullable in the fused variant (only q_out wanted)
  float* q_scale;
  // Fused variant only (RMSNorm and RoPE on Q / K before the quantization).
  const int32_t* positions;  // [T], needed when rd > 0
  const float* cos_sin;      // [max_pos, rd]: cos of the rd/2 frequencies, then their sin
  int max_pos, rd;           // rd = 0: no rotation
  const uint16_t* q_norm_w;  // [D] bf16, nullable
  const uint16_t* k_norm_w;  // [D] bf16, nullable
  float eps;
  uint16_t* q_out;  // [T, Hq, D] bf16, nullable
  uint16_t* k_out;  // [T, Hkv, D] bf16, nullable
  const float* k_smooth;  // [Hkv, D] per-channel K smoothing factors, nullable
};

// Decode (INT8 and BF16-KV variants share the work split and the workspace).
struct DecodeParams {
  void* out;                  // [B, Hq, D], fp32 or (out_bf16) bf16
  int out_bf16;
  const void* q;              // int8 [B, Hq, D] (INT8 path) or bf16 [B, Hq, D] (BF16 path)
  const float* q_scale;       // [B, Hq] (INT8 path)
  const void* k_cache;
  const void* v_cache;
  const float* k_scale;       // INT8 path
  const float* v_scale;
  const int32_t* block_tables;  // [B, max_blocks]
  const int32_t* seq_lens;      // [B]
  int B, Hq, Hkv, G, D, max_blocks, num_blocks;
  float sm_scale;
  float* ws_part;             // [(B*Hkv + grid) slots][8 rows * D + 16]
  int grid;                   // CTAs launched (the work split depends on it)
  // Decode step (INT8 path, step != 0): the newest token of each sequence
  // (position seq_lens[b] - 1) arrives as bf16 and is quantized inside the
  // kernel -- K/V written into the cache, Q quantized per warp -- instead of
  // being read from q / the cache.
  int step;
  int u8_probs;               // INT8 path: probability codes 0..255 (sW = A / 255) instead of 0..127
  const uint16_t* q_bf16;     // [B, Hq, D]
  const uint16_t* k_new;      // [B, Hkv, D]
  const uint16_t* v_new;      // [B, Hkv, D]
  int8_t* k_cache_w;          // the caches again, written at the new token's slot
  int8_t* v_cache_w;
  float* k_scale_w;
  float* v_scale_w;
};

// Debug QK: int32 accumulators through the decode kernel's QK fragments.
struct DebugQKParams {
  int32_t* acc;               // [B, Hq, max_len]
  const int8_t* q;            // [B, Hq, D]
  const int8_t* k_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  int B, Hq, Hkv, G, D, max_blocks, num_blocks, max_len;
};

struct PrefixParams {
  void* out;                  // [C, Hq, D], fp32 or (out_bf16) bf16
  const int8_t* q;            // [C, Hq, D]
  const float* q_scale;       // [C, Hq]
  const int8_t* k_cache;
  const int8_t* v_cache;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_table;
  int H, C, Hq, Hkv, G, D, num_blocks;
  float sm_scale;
  uint8_t* tiles;  // workspace: f16 (bf16) operand tiles per (KV head, 32-key group)
  // High-precision variant: bf16 query and the chunk's own bf16 K/V (the
  // history still comes from the INT8 cache, read back as code x scale).
  const uint16_t* qb;       // [C, Hq, D]
  const uint16_t* k_chunk;  // [C, Hkv, D]
  const uint16_t* v_chunk;  // [C, Hkv, D]
  // Work items (set by the launcher): row blocks (128 rows of one KV head) in
  // order of decreasing cost; the first full_items run whole, each of the rest
  // is split into split_k parts over its key groups, whose (o, m, l) go to part
  // and are merged by a second kernel.
  int nrb, full_items, split_k;
  float* part;  // [split items][128 rows][D + 2]
  int out_bf16;
  // Debug record (i8kv_debug_prefix_i32): S [C, Hq, H + C], Wq [C, Hq, NG * 32]
  // and PV [C, Hq, NG, D] with NG = ceil((H + C) / 32).
  int32_t* dbg_s;
  uint8_t* dbg_wq;
  int32_t* dbg_pv;
  // BF16-KV comparison: every key (history and chunk) from the bf16 paged cache
  const uint16_t* kb_cache;  // [NB, Hkv, D/8, 16, 8]
  const uint16_t* vb_cache;  // [NB, Hkv, D, 16]
};

// Per-translation-unit device error words (read and cleared).
cudaError_t read_error_producer(int* value);
cudaError_t read_error_decode(int* value);
cudaError_t read_error_prefix(int* value);

cudaError_t launch_kv_quant_write(const ProducerParams& p, cudaStream_t stream);
cudaError_t launch_kv_rope_quant_write(const ProducerParams& p, cudaStream_t stream);
size_t prefix_workspace_bytes(int H, int C, int Hkv, int D);
cudaError_t launch_bf16_kv_write(const ProducerParams& p, uint16_t* k_cache, uint16_t* v_cache, cudaStream_t stream);

// Per-device decode geometry: CTAs per launch and dynamic shared memory.
int decode_grid(int device, int B, int Hkv, int max_blocks);
size_t decode_workspace_bytes(int B, int Hkv, int D, int grid);
cudaError_t launch_int8_decode(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_bf16_decode(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_debug_qk(const DebugQKParams& p, cudaStream_t stream);

// Fixed device scratch of the allocation-free decode entry point (decode.cu).
size_t noalloc_scratch_bytes();
// Device address of that scratch in the calling thread's current context
// (looked up once per context and cached).
cudaError_t noalloc_scratch_address(void** addr);
cudaError_t launch_int8_prefix(const PrefixParams& p, cudaStream_t stream);
cudaError_t launch_bf16_prefix(const PrefixParams& p, cudaStream_t stream);
cudaError_t launch_debug_prefix(const PrefixParams& p, cudaStream_t stream);

}  // namespace i8kv
