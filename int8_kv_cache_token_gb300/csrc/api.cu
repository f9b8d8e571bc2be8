// api.cu -- the extern "C" boundary declared in include/i8kv.h: argument
// checking, status codes, the last-error string and the launches.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/i8kv.h"
#include "kernels.h"

namespace {

thread_local std::string g_last_error;

i8kv_status fail(i8kv_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));

i8kv_status fail(i8kv_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

i8kv_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return I8KV_OK;
  return fail(I8KV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQUIRE(cond, status, ...) \
  do {                             \
    if (!(cond)) return fail(status, __VA_ARGS__); \
  } while (0)

i8kv_status check_heads(int Hq, int Hkv, int D) {
  REQUIRE(Hq > 0 && Hkv > 0, I8KV_ERR_INVALID_ARG, "Hq=%d Hkv=%d must be positive", Hq, Hkv);
  REQUIRE(Hq % Hkv == 0, I8KV_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  REQUIRE(Hq / Hkv <= 8, I8KV_ERR_UNSUPPORTED, "G=Hq/Hkv=%d > 8 is not supported", Hq / Hkv);
  REQUIRE(D == 128 || D == 256, I8KV_ERR_UNSUPPORTED, "head_dim %d not supported (128 or 256)", D);
  REQUIRE(Hkv <= 8, I8KV_ERR_UNSUPPORTED, "Hkv=%d > 8 is not supported", Hkv);
  return I8KV_OK;
}

i8kv_status check_out(const void* out, int out_dtype) {
  REQUIRE(out_dtype == I8KV_OUT_F32 || out_dtype == I8KV_OUT_BF16, I8KV_ERR_INVALID_ARG,
          "out_dtype=%d (I8KV_OUT_F32 or I8KV_OUT_BF16)", out_dtype);
  REQUIRE(out != nullptr, I8KV_ERR_INVALID_ARG, "out is NULL");
  REQUIRE(aligned16(out), I8KV_ERR_INVALID_ARG, "out must be 16-byte aligned");
  return I8KV_OK;
}

}  // namespace

extern "C" {

i8kv_status i8kv_last_error(char* buf, size_t n) {
  if (buf && n) {
    std::strncpy(buf, g_last_error.c_str(), n - 1);
    buf[n - 1] = '\0';
  }
  return I8KV_OK;
}

i8kv_status i8kv_device_error(int* code) {
  REQUIRE(code != nullptr, I8KV_ERR_INVALID_ARG, "code is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return from_cuda(e, "i8kv_device_error: synchronize");
  int v = 0;
  cudaError_t (*readers[])(int*) = {i8kv::read_error_producer, i8kv::read_error_decode, i8kv::read_error_prefix};
  for (auto rd : readers) {
    int x = 0;
    e = rd(&x);
    if (e != cudaSuccess) return from_cuda(e, "i8kv_device_error: read");
    if (v == 0) v = x;
  }
  *code = v;
  if (v != 0) return fail(I8KV_ERR_DEVICE, "a kernel recorded device error %d", v);
  return I8KV_OK;
}

int i8kv_version(void) { return 100; }

i8kv_status i8kv_kv_quant_write(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping, int T, int Hkv,
                                int D, int block_size, int num_blocks, int8_t* k_cache, int8_t* v_cache,
                                float* k_scale, float* v_scale, const uint16_t* q, int Hq, int8_t* q_i8,
                                float* q_scale, void* stream) {
  REQUIRE(T >= 0, I8KV_ERR_INVALID_ARG, "T=%d < 0", T);
  REQUIRE(block_size == 16, I8KV_ERR_UNSUPPORTED, "block_size %d not supported (16)", block_size);
  REQUIRE(D == 128 || D == 256, I8KV_ERR_UNSUPPORTED, "head_dim %d not supported (128 or 256)", D);
  REQUIRE(Hkv > 0 && Hkv <= 8, I8KV_ERR_UNSUPPORTED, "Hkv=%d not in 1..8", Hkv);
  REQUIRE(num_blocks > 0, I8KV_ERR_INVALID_ARG, "num_blocks=%d", num_blocks);
  if (T == 0) return I8KV_OK;
  REQUIRE(k && v && slot_mapping && k_cache && v_cache && k_scale && v_scale, I8KV_ERR_INVALID_ARG,
          "null K/V/slot/cache/scale pointer");
  REQUIRE(aligned16(k) && aligned16(v) && aligned16(k_cache) && aligned16(v_cache), I8KV_ERR_INVALID_ARG,
          "K/V inputs and caches must be 16-byte aligned");
  if (q) {
    REQUIRE(Hq > 0, I8KV_ERR_INVALID_ARG, "Hq=%d with a query", Hq);
    REQUIRE(q_i8 && q_scale, I8KV_ERR_INVALID_ARG, "q given without q_i8/q_scale");
    REQUIRE(aligned16(q) && aligned16(q_i8), I8KV_ERR_INVALID_ARG, "q and q_i8 must be 16-byte aligned");
  }
  i8kv::ProducerParams p{k, v, slot_mapping, T, Hkv, D, num_blocks, k_cache, v_cache, k_scale, v_scale,
                         q, q ? Hq : 0, q_i8, q_scale};
  return from_cuda(i8kv::launch_kv_quant_write(p, static_cast<cudaStream_t>(stream)), "kv_quant_write launch");
}

i8kv_status i8kv_kv_rope_quant_write(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping, int T,
                                     int Hkv, int D, int block_size, int num_blocks, int8_t* k_cache, int8_t* v_cache,
                                     float* k_scale, float* v_scale, const uint16_t* q, int Hq, int8_t* q_i8,
                                     float* q_scale, const int32_t* positions, const float* cos_sin, int max_position,
                                     int rotary_dim, const uint16_t* q_norm_weight, const uint16_t* k_norm_weight,
                                     float norm_eps, uint16_t* q_out, uint16_t* k_out, const float* k_smooth,
                                     void* stream) {
  REQUIRE(T >= 0, I8KV_ERR_INVALID_ARG, "T=%d < 0", T);
  REQUIRE(block_size == 16, I8KV_ERR_UNSUPPORTED, "block_size %d not supported (16)", block_size);
  REQUIRE(D == 128 || D == 256, I8KV_ERR_UNSUPPORTED, "head_dim %d not supported (128 or 256)", D);
  REQUIRE(Hkv > 0 && Hkv <= 8, I8KV_ERR_UNSUPPORTED, "Hkv=%d not in 1..8", Hkv);
  REQUIRE(num_blocks > 0, I8KV_ERR_INVALID_ARG, "num_blocks=%d", num_blocks);
  REQUIRE(rotary_dim >= 0 && rotary_dim <= D, I8KV_ERR_INVALID_ARG, "rotary_dim=%d not in 0..%d", rotary_dim, D);
  REQUIRE(rotary_dim % 32 == 0, I8KV_ERR_UNSUPPORTED, "rotary_dim=%d not a multiple of 32", rotary_dim);
  if (rotary_dim > 0) {
    REQUIRE(positions && cos_sin, I8KV_ERR_INVALID_ARG, "rotary_dim > 0 needs positions and cos_sin");
    REQUIRE(max_position > 0, I8KV_ERR_INVALID_ARG, "max_position=%d", max_position);
    REQUIRE(aligned16(cos_sin), I8KV_ERR_INVALID_ARG, "cos_sin must be 16-byte aligned");
  }
  if (q_norm_weight || k_norm_weight) {
    REQUIRE(norm_eps > 0.f && norm_eps < 3.0e38f, I8KV_ERR_INVALID_ARG, "norm_eps must be positive and finite");
    REQUIRE(aligned16(q_norm_weight) && aligned16(k_norm_weight), I8KV_ERR_INVALID_ARG,
            "norm weights must be 16-byte aligned");
  }
  if (k_smooth) {
    REQUIRE(aligned16(k_smooth), I8KV_ERR_INVALID_ARG, "k_smooth must be 16-byte aligned");
    REQUIRE(!q || (Hq > 0 && Hq % Hkv == 0), I8KV_ERR_INVALID_ARG, "k_smooth needs Hq a multiple of Hkv");
  }
  if (T == 0) return I8KV_OK;
  REQUIRE(k && v && slot_mapping && k_cache && v_cache && k_scale && v_scale, I8KV_ERR_INVALID_ARG,
          "null K/V/slot/cache/scale pointer");
  REQUIRE(aligned16(k) && aligned16(v) && aligned16(k_cache) && aligned16(v_cache) && aligned16(k_out),
          I8KV_ERR_INVALID_ARG, "K/V inputs, caches and k_out must be 16-byte aligned");
  REQUIRE(q || !q_out, I8KV_ERR_INVALID_ARG, "q_out given without q");
  if (q) {
    REQUIRE(Hq > 0, I8KV_ERR_INVALID_ARG, "Hq=%d with a query", Hq);
    REQUIRE((q_i8 != nullptr) == (q_scale != nullptr), I8KV_ERR_INVALID_ARG, "q_i8 and q_scale go together");
    REQUIRE(q_i8 || q_out, I8KV_ERR_INVALID_ARG, "q given without q_i8/q_scale or q_out");
    REQUIRE(aligned16(q) && aligned16(q_i8) && aligned16(q_out), I8KV_ERR_INVALID_ARG,
            "q, q_i8 and q_out must be 16-byte aligned");
  }
  i8kv::ProducerParams p{k, v, slot_mapping, T, Hkv, D, num_blocks, k_cache, v_cache, k_scale, v_scale,
                         q, q ? Hq : 0, q_i8, q_scale};
  p.positions = rotary_dim > 0 ? positions : nullptr;
  p.cos_sin = rotary_dim > 0 ? cos_sin : nullptr;
  p.max_pos = max_position;
  p.rd = rotary_dim;
  p.q_norm_w = q_norm_weight;
  p.k_norm_w = k_norm_weight;
  p.eps = norm_eps;
  p.q_out = q_out;
  p.k_out = k_out;
  p.k_smooth = k_smooth;
  return from_cuda(i8kv::launch_kv_rope_quant_write(p, static_cast<cudaStream_t>(stream)),
                   "kv_rope_quant_write launch");
}

size_t i8kv_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int max_blocks, int block_size, int partition) {
  (void)Hq;
  (void)block_size;
  (void)partition;
  if (B <= 0 || Hkv <= 0 || max_blocks <= 0 || (D != 128 && D != 256)) return 0;
  int dev = 0;
  cudaGetDevice(&dev);
  return i8kv::decode_workspace_bytes(B, Hkv, D, i8kv::decode_grid(dev, B, Hkv, max_blocks));
}

static i8kv_status decode_common(i8kv::DecodeParams& p, const void* q, const float* q_scale, bool int8,
                                 const void* k_cache, const void* v_cache, const float* k_scale,
                                 const float* v_scale, const int32_t* block_tables, const int32_t* seq_lens, int B,
                                 int Hq, int Hkv, int D, int block_size, int max_blocks, int num_blocks,
                                 float softmax_scale, int partition, void* workspace, size_t workspace_bytes,
                                 void* out, int out_dtype) {
  REQUIRE(B >= 0, I8KV_ERR_INVALID_ARG, "B=%d < 0", B);
  i8kv_status s = check_heads(Hq, Hkv, D);
  if (s != I8KV_OK) return s;
  s = check_out(out, out_dtype);
  if (s != I8KV_OK) return s;
  REQUIRE(block_size == 16, I8KV_ERR_UNSUPPORTED, "block_size %d not supported (16)", block_size);
  REQUIRE(partition == 256, I8KV_ERR_UNSUPPORTED, "partition %d not supported (256)", partition);
  REQUIRE(max_blocks > 0 && num_blocks > 0, I8KV_ERR_INVALID_ARG, "max_blocks=%d num_blocks=%d", max_blocks,
          num_blocks);
  REQUIRE(out && q && k_cache && v_cache && block_tables && seq_lens, I8KV_ERR_INVALID_ARG, "null pointer");
  if (int8) REQUIRE(k_scale && v_scale, I8KV_ERR_INVALID_ARG, "null scale pointer");
  REQUIRE(aligned16(k_cache) && aligned16(v_cache) && aligned16(q), I8KV_ERR_INVALID_ARG,
          "caches and q must be 16-byte aligned");
  if (int8) REQUIRE(aligned16(k_scale) && aligned16(v_scale), I8KV_ERR_INVALID_ARG, "scales must be 16-byte aligned");
  int dev = 0;
  cudaGetDevice(&dev);
  const int grid = i8kv::decode_grid(dev, B, Hkv, max_blocks);
  const size_t need = i8kv::decode_workspace_bytes(B, Hkv, D, grid);
  REQUIRE(workspace != nullptr && workspace_bytes >= need, I8KV_ERR_WORKSPACE,
          "workspace of %zu bytes given, %zu needed", workspace_bytes, need);
  REQUIRE(aligned16(workspace), I8KV_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  float* ws = static_cast<float*>(workspace);
  p.out = out;
  p.out_bf16 = out_dtype == I8KV_OUT_BF16;
  p.q = q;
  p.q_scale = q_scale;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.D = D;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.sm_scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
  p.ws_part = ws;
  p.grid = grid;
  return I8KV_OK;
}

i8kv_status i8kv_int8_paged_decode_attn(void* out, int out_dtype, const int8_t* q_i8, const float* q_scale,
                                        const int8_t* k_cache,
                                        const int8_t* v_cache, const float* k_scale, const float* v_scale,
                                        const int32_t* block_tables, const int32_t* seq_lens, int B, int Hq, int Hkv,
                                        int D, int block_size, int max_blocks, int num_blocks, float softmax_scale,
                                        int partition, void* workspace, size_t workspace_bytes, void* stream) {
  REQUIRE(q_scale != nullptr, I8KV_ERR_INVALID_ARG, "q_scale is NULL");
  i8kv::DecodeParams p{};
  i8kv_status s = decode_common(p, q_i8, q_scale, true, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                                B, Hq, Hkv, D, block_size, max_blocks, num_blocks, softmax_scale, partition,
                                workspace, workspace_bytes, out, out_dtype);
  if (s != I8KV_OK || B == 0) return s;
  return from_cuda(i8kv::launch_int8_decode(p, static_cast<cudaStream_t>(stream)), "int8 decode launch");
}

i8kv_status i8kv_int8_paged_decode_attn_u8p(void* out, int out_dtype, const int8_t* q_i8, const float* q_scale,
                                            const int8_t* k_cache, const int8_t* v_cache, const float* k_scale,
                                            const float* v_scale, const int32_t* block_tables,
                                            const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int block_size,
                                            int max_blocks, int num_blocks, float softmax_scale, int partition,
                                            void* workspace, size_t workspace_bytes, void* stream) {
  REQUIRE(q_scale != nullptr, I8KV_ERR_INVALID_ARG, "q_scale is NULL");
  i8kv::DecodeParams p{};
  i8kv_status s = decode_common(p, q_i8, q_scale, true, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                                B, Hq, Hkv, D, block_size, max_blocks, num_blocks, softmax_scale, partition,
                                workspace, workspace_bytes, out, out_dtype);
  if (s != I8KV_OK || B == 0) return s;
  p.u8_probs = 1;
  return from_cuda(i8kv::launch_int8_decode(p, static_cast<cudaStream_t>(stream)), "int8 decode (u8 P) launch");
}

i8kv_status i8kv_int8_decode_step(void* out, int out_dtype, const uint16_t* q, const uint16_t* k_new,
                                  const uint16_t* v_new,
                                  int8_t* k_cache, int8_t* v_cache, float* k_scale, float* v_scale,
                                  const int32_t* block_tables, const int32_t* seq_lens, int B, int Hq, int Hkv, int D,
                                  int block_size, int max_blocks, int num_blocks, float softmax_scale, int partition,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  REQUIRE(k_new && v_new, I8KV_ERR_INVALID_ARG, "k_new / v_new is NULL");
  REQUIRE(aligned16(k_new) && aligned16(v_new), I8KV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  i8kv::DecodeParams p{};
  i8kv_status s = decode_common(p, q, nullptr, true, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, B,
                                Hq, Hkv, D, block_size, max_blocks, num_blocks, softmax_scale, partition, workspace,
                                workspace_bytes, out, out_dtype);
  if (s != I8KV_OK || B == 0) return s;
  p.step = 1;
  p.q_bf16 = q;
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_cache_w = k_cache;
  p.v_cache_w = v_cache;
  p.k_scale_w = k_scale;
  p.v_scale_w = v_scale;
  return from_cuda(i8kv::launch_int8_decode(p, static_cast<cudaStream_t>(stream)), "int8 decode step launch");
}

i8kv_status i8kv_int8_paged_decode_attn_noalloc(float* out, const int8_t* q_i8, const float* q_scale,
                                                const int8_t* k_cache, const int8_t* v_cache, const float* k_scale,
                                                const float* v_scale, const int32_t* block_tables,
                                                const int32_t* seq_lens, int B, int Hq, int Hkv, int D,
                                                int block_size, int max_blocks, int num_blocks, float softmax_scale,
                                                int partition, void* stream) {
  // Same checks and the same kernel as i8kv_int8_paged_decode_attn; only the
  // workspace comes from the library's fixed device scratch instead of the caller.
  i8kv_status s = check_heads(Hq, Hkv, D);
  if (s != I8KV_OK) return s;
  REQUIRE(B >= 0 && max_blocks > 0, I8KV_ERR_INVALID_ARG, "B=%d max_blocks=%d", B, max_blocks);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e, "noalloc decode: cudaGetDevice");
  const int grid = i8kv::decode_grid(dev, B, Hkv, max_blocks);
  const size_t need = i8kv::decode_workspace_bytes(B, Hkv, D, grid);
  REQUIRE(need <= i8kv::noalloc_scratch_bytes(), I8KV_ERR_WORKSPACE,
          "noalloc decode needs %zu bytes of scratch for B=%d Hkv=%d D=%d; the fixed scratch holds %zu bytes "
          "(use i8kv_int8_paged_decode_attn with a caller workspace)",
          need, B, Hkv, D, i8kv::noalloc_scratch_bytes());
  void* scratch = nullptr;
  e = i8kv::noalloc_scratch_address(&scratch);
  if (e != cudaSuccess) return from_cuda(e, "noalloc decode: cudaGetSymbolAddress");
  i8kv::DecodeParams p{};
  s = decode_common(p, q_i8, q_scale, true, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, B, Hq, Hkv,
                    D, block_size, max_blocks, num_blocks, softmax_scale, partition, scratch, need, out,
                    I8KV_OUT_F32);
  if (s != I8KV_OK || B == 0) return s;
  return from_cuda(i8kv::launch_int8_decode(p, static_cast<cudaStream_t>(stream)), "noalloc int8 decode launch");
}

size_t i8kv_prefix_workspace_bytes(int history_len, int chunk_len, int Hkv, int D) {
  if (history_len < 0 || chunk_len <= 0 || Hkv <= 0 || (D != 128 && D != 256)) return 0;
  return i8kv::prefix_workspace_bytes(history_len, chunk_len, Hkv, D);
}

i8kv_status i8kv_int8_prefix_attn(void* out, int out_dtype, const int8_t* q_i8, const float* q_scale,
                                  const int8_t* k_cache,
                                  const int8_t* v_cache, const float* k_scale, const float* v_scale,
                                  const int32_t* block_table, int history_len, int chunk_len, int Hq, int Hkv, int D,
                                  int block_size, int num_blocks, float softmax_scale, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  REQUIRE(history_len >= 0 && chunk_len >= 0, I8KV_ERR_INVALID_ARG, "history_len=%d chunk_len=%d", history_len,
          chunk_len);
  i8kv_status s = check_heads(Hq, Hkv, D);
  if (s != I8KV_OK) return s;
  REQUIRE(block_size == 16, I8KV_ERR_UNSUPPORTED, "block_size %d not supported (16)", block_size);
  REQUIRE(num_blocks > 0, I8KV_ERR_INVALID_ARG, "num_blocks=%d", num_blocks);
  if (chunk_len == 0) return I8KV_OK;
  s = check_out(out, out_dtype);
  if (s != I8KV_OK) return s;
  REQUIRE(q_i8 && q_scale && k_cache && v_cache && k_scale && v_scale && block_table, I8KV_ERR_INVALID_ARG,
          "null pointer");
  REQUIRE(aligned16(k_cache) && aligned16(v_cache) && aligned16(q_i8) && aligned16(k_scale) && aligned16(v_scale),
          I8KV_ERR_INVALID_ARG, "caches, scales and q must be 16-byte aligned");
  const size_t need = i8kv::prefix_workspace_bytes(history_len, chunk_len, Hkv, D);
  REQUIRE(workspace != nullptr && workspace_bytes >= need, I8KV_ERR_WORKSPACE,
          "prefix workspace of %zu bytes given, %zu needed", workspace_bytes, need);
  REQUIRE(aligned16(workspace), I8KV_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  i8kv::PrefixParams p{out, q_i8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, history_len, chunk_len,
                       Hq, Hkv, Hq / Hkv, D, num_blocks, softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D),
                       static_cast<uint8_t*>(workspace)};
  p.out_bf16 = out_dtype == I8KV_OUT_BF16;
  return from_cuda(i8kv::launch_int8_prefix(p, static_cast<cudaStream_t>(stream)), "int8 prefix launch");
}

i8kv_status i8kv_bf16_prefix_attn(void* out, int out_dtype, const uint16_t* q, const uint16_t* k_chunk,
                                  const uint16_t* v_chunk,
                                  const int8_t* k_cache, const int8_t* v_cache, const float* k_scale,
                                  const float* v_scale, const int32_t* block_table, int history_len, int chunk_len,
                                  int Hq, int Hkv, int D, int block_size, int num_blocks, float softmax_scale,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  REQUIRE(history_len >= 0 && chunk_len >= 0, I8KV_ERR_INVALID_ARG, "history_len=%d chunk_len=%d", history_len,
          chunk_len);
  i8kv_status s = check_heads(Hq, Hkv, D);
  if (s != I8KV_OK) return s;
  REQUIRE(block_size == 16, I8KV_ERR_UNSUPPORTED, "block_size %d not supported (16)", block_size);
  if (chunk_len == 0) return I8KV_OK;
  s = check_out(out, out_dtype);
  if (s != I8KV_OK) return s;
  REQUIRE(q && k_chunk && v_chunk, I8KV_ERR_INVALID_ARG, "null q/k_chunk/v_chunk pointer");
  REQUIRE(aligned16(q) && aligned16(k_chunk) && aligned16(v_chunk), I8KV_ERR_INVALID_ARG,
          "q, k_chunk and v_chunk must be 16-byte aligned");
  if (history_len > 0) {
    REQUIRE(num_blocks > 0, I8KV_ERR_INVALID_ARG, "num_blocks=%d", num_blocks);
    REQUIRE(k_cache && v_cache && k_scale && v_scale && block_table, I8KV_ERR_INVALID_ARG,
            "history_len > 0 needs the caches, scales and block_table");
    REQUIRE(aligned16(k_cache) && aligned16(v_cache), I8KV_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  }
  const size_t need = i8kv::prefix_workspace_bytes(history_len, chunk_len, Hkv, D);
  REQUIRE(workspace != nullptr && workspace_bytes >= need, I8KV_ERR_WORKSPACE,
          "prefix workspace of %zu bytes given, %zu needed", workspace_bytes, need);
  REQUIRE(aligned16(workspace), I8KV_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  i8kv::PrefixParams p{out, nullptr, nullptr, k_cache, v_cache, k_scale, v_scale, block_table, history_len, chunk_len,
                       Hq, Hkv, Hq / Hkv, D, num_blocks, softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D),
                       static_cast<uint8_t*>(workspace)};
  p.qb = q;
  p.k_chunk = k_chunk;
  p.v_chunk = v_chunk;
  p.out_bf16 = out_dtype == I8KV_OUT_BF16;
  return from_cuda(i8kv::launch_bf16_prefix(p, static_cast<cudaStream_t>(stream)), "bf16 prefix launch");
}

i8kv_status i8kv_bf16_kv_prefix_attn(void* out, int out_dtype, const uint16_t* q, const uint16_t* k_cache,
                                     const uint16_t* v_cache, const int32_t* block_table, int history_len,
                                     int chunk_len, int Hq, int Hkv, int D, int block_size, int num_blocks,
                                     float softmax_scale, void* workspace, size_t workspace_bytes, void* stream) {
  REQUIRE(history_len >= 0 && chunk_len >= 0, I8KV_ERR_INVALID_ARG, "history_len=%d chunk_len=%d", history_len,
          chunk_len);
  i8kv_status s = check_heads(Hq, Hkv, D);
  if (s != I8KV_OK) return s;
  REQUIRE(block_size == 16, I8KV_ERR_UNSUPPORTED, "block_size %d not supported (16)", block_size);
  REQUIRE(num_blocks > 0, I8KV_ERR_INVALID_ARG, "num_blocks=%d", num_blocks);
  if (chunk_len == 0) return I8KV_OK;
  s = check_out(out, out_dtype);
  if (s != I8KV_OK) return s;
  REQUIRE(q && k_cache && v_cache && block_table, I8KV_ERR_INVALID_ARG, "null q/cache/block_table pointer");
  REQUIRE(aligned16(q) && aligned16(k_cache) && aligned16(v_cache), I8KV_ERR_INVALID_ARG,
          "q and the caches must be 16-byte aligned");
  const size_t need = i8kv::prefix_workspace_bytes(history_len, chunk_len, Hkv, D);
  REQUIRE(workspace != nullptr && workspace_bytes >= need, I8KV_ERR_WORKSPACE,
          "prefix workspace of %zu bytes given, %zu needed", workspace_bytes, need);
  REQUIRE(aligned16(workspace), I8KV_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  i8kv::PrefixParams p{out, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, block_table, history_len,
                       chunk_len, Hq, Hkv, Hq / Hkv, D, num_blocks,
                       softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D), static_cast<uint8_t*>(workspace)};
  p.qb = q;
  p.kb_cache = k_cache;
  p.vb_cache = v_cache;
  p.out_bf16 = out_dtype == I8KV_OUT_BF16;
  return from_cuda(i8kv::launch_bf16_prefix(p, static_cast<cudaStream_t>(stream)), "bf16-kv prefix launch");
}

i8kv_status i8kv_prefill_chunk(void* out, int out_dtype, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const int32_t* slot_mapping, int8_t* k_cache, int8_t* v_cache, float* k_scale,
                               float* v_scale, const int32_t* block_table, int history_len, int chunk_len, int Hq,
                               int Hkv, int D, int block_size, int num_blocks, int int8_min_history,
                               float softmax_scale, int8_t* q_i8, float* q_scale, void* workspace,
                               size_t workspace_bytes, int* route, void* stream) {
  REQUIRE(history_len >= 0 && chunk_len >= 0, I8KV_ERR_INVALID_ARG, "history_len=%d chunk_len=%d", history_len,
          chunk_len);
  i8kv_status s = check_heads(Hq, Hkv, D);
  if (s != I8KV_OK) return s;
  const bool int8 = history_len >= int8_min_history;
  if (route) *route = int8 ? I8KV_ROUTE_INT8 : I8KV_ROUTE_BF16;
  if (chunk_len == 0) return I8KV_OK;
  s = check_out(out, out_dtype);
  if (s != I8KV_OK) return s;
  REQUIRE(q && block_table && k_cache && v_cache && k_scale && v_scale, I8KV_ERR_INVALID_ARG,
          "null q/block_table/cache pointer");
  if (int8) REQUIRE(q_i8 && q_scale, I8KV_ERR_INVALID_ARG, "the INT8 route needs q_i8 and q_scale");
  const size_t need = i8kv::prefix_workspace_bytes(history_len, chunk_len, Hkv, D);
  REQUIRE(workspace != nullptr && workspace_bytes >= need, I8KV_ERR_WORKSPACE,
          "prefix workspace of %zu bytes given, %zu needed", workspace_bytes, need);
  // the chunk's K/V (and, on the INT8 route, its query) through the producer
  s = i8kv_kv_quant_write(k, v, slot_mapping, chunk_len, Hkv, D, block_size, num_blocks, k_cache, v_cache, k_scale,
                          v_scale, int8 ? q : nullptr, Hq, q_i8, q_scale, stream);
  if (s != I8KV_OK) return s;
  if (int8)
    return i8kv_int8_prefix_attn(out, out_dtype, q_i8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, history_len,
                                 chunk_len, Hq, Hkv, D, block_size, num_blocks, softmax_scale, workspace,
                                 workspace_bytes, stream);
  return i8kv_bf16_prefix_attn(out, out_dtype, q, k, v, k_cache, v_cache, k_scale, v_scale, block_table, history_len, chunk_len,
                               Hq, Hkv, D, block_size, num_blocks, softmax_scale, workspace, workspace_bytes, stream);
}

i8kv_status i8kv_debug_prefix_i32(int32_t* s_acc, uint8_t* wq, int32_t* pv_acc, float* out, const int8_t* q_i8,
                                  const float* q_scale, const int8_t* k_cache, const int8_t* v_cache,
                                  const float* k_scale, const float* v_scale, const int32_t* block_table,
                                  int history_len, int chunk_len, int Hq, int Hkv, int D, int block_size,
                                  int num_blocks, float softmax_scale, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  REQUIRE(history_len >= 0 && chunk_len >= 0, I8KV_ERR_INVALID_ARG, "history_len=%d chunk_len=%d", history_len,
          chunk_len);
  i8kv_status s = check_heads(Hq, Hkv, D);
  if (s != I8KV_OK) return s;
  REQUIRE(block_size == 16, I8KV_ERR_UNSUPPORTED, "block_size %d not supported (16)", block_size);
  REQUIRE(num_blocks > 0, I8KV_ERR_INVALID_ARG, "num_blocks=%d", num_blocks);
  if (chunk_len == 0) return I8KV_OK;
  s = check_out(out, I8KV_OUT_F32);
  if (s != I8KV_OK) return s;
  REQUIRE(s_acc && wq && pv_acc && q_i8 && q_scale && k_cache && v_cache && k_scale && v_scale && block_table,
          I8KV_ERR_INVALID_ARG, "null pointer");
  REQUIRE(aligned16(k_cache) && aligned16(v_cache) && aligned16(q_i8) && aligned16(k_scale) && aligned16(v_scale),
          I8KV_ERR_INVALID_ARG, "caches, scales and q must be 16-byte aligned");
  const size_t need = i8kv::prefix_workspace_bytes(history_len, chunk_len, Hkv, D);
  REQUIRE(workspace != nullptr && workspace_bytes >= need, I8KV_ERR_WORKSPACE,
          "prefix workspace of %zu bytes given, %zu needed", workspace_bytes, need);
  REQUIRE(aligned16(workspace), I8KV_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  i8kv::PrefixParams p{out, q_i8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, history_len, chunk_len,
                       Hq, Hkv, Hq / Hkv, D, num_blocks, softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D),
                       static_cast<uint8_t*>(workspace)};
  p.dbg_s = s_acc;
  p.dbg_wq = wq;
  p.dbg_pv = pv_acc;
  return from_cuda(i8kv::launch_debug_prefix(p, static_cast<cudaStream_t>(stream)), "debug prefix launch");
}

i8kv_status i8kv_debug_qk_i32(int32_t* acc, const int8_t* q_i8, const int8_t* k_cache, const int32_t* block_tables,
                              const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int block_size, int max_blocks,
                              int num_blocks, int max_len, void* stream) {
  REQUIRE(B >= 0 && max_len >= 0, I8KV_ERR_INVALID_ARG, "B=%d max_len=%d", B, max_len);
  i8kv_status s = check_heads(Hq, Hkv, D);
  if (s != I8KV_OK) return s;
  REQUIRE(block_size == 16, I8KV_ERR_UNSUPPORTED, "block_size %d not supported (16)", block_size);
  REQUIRE(max_blocks > 0 && num_blocks > 0, I8KV_ERR_INVALID_ARG, "max_blocks=%d num_blocks=%d", max_blocks,
          num_blocks);
  if (B == 0 || max_len == 0) return I8KV_OK;
  REQUIRE(acc && q_i8 && k_cache && block_tables && seq_lens, I8KV_ERR_INVALID_ARG, "null pointer");
  REQUIRE(aligned16(k_cache) && aligned16(q_i8), I8KV_ERR_INVALID_ARG, "k_cache and q must be 16-byte aligned");
  i8kv::DebugQKParams p{acc, q_i8, k_cache, block_tables, seq_lens, B, Hq, Hkv, Hq / Hkv, D, max_blocks, num_blocks,
                        max_len};
  return from_cuda(i8kv::launch_debug_qk(p, static_cast<cudaStream_t>(stream)), "debug qk launch");
}

i8kv_status i8kv_bf16_kv_write(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping, int T, int Hkv,
                               int D, int block_size, int num_blocks, uint16_t* k_cache, uint16_t* v_cache,
                               void* stream) {
  REQUIRE(T >= 0, I8KV_ERR_INVALID_ARG, "T=%d < 0", T);
  REQUIRE(block_size == 16, I8KV_ERR_UNSUPPORTED, "block_size %d not supported (16)", block_size);
  REQUIRE(D == 128 || D == 256, I8KV_ERR_UNSUPPORTED, "head_dim %d not supported (128 or 256)", D);
  REQUIRE(Hkv > 0, I8KV_ERR_INVALID_ARG, "Hkv=%d", Hkv);
  REQUIRE(num_blocks > 0, I8KV_ERR_INVALID_ARG, "num_blocks=%d", num_blocks);
  if (T == 0) return I8KV_OK;
  REQUIRE(k && v && slot_mapping && k_cache && v_cache, I8KV_ERR_INVALID_ARG, "null pointer");
  REQUIRE(aligned16(k) && aligned16(v) && aligned16(k_cache) && aligned16(v_cache), I8KV_ERR_INVALID_ARG,
          "K/V inputs and caches must be 16-byte aligned");
  i8kv::ProducerParams p{k, v, slot_mapping, T, Hkv, D, num_blocks, nullptr, nullptr, nullptr, nullptr,
                         nullptr, 0, nullptr, nullptr};
  return from_cuda(i8kv::launch_bf16_kv_write(p, k_cache, v_cache, static_cast<cudaStream_t>(stream)),
                   "bf16 kv write launch");
}

i8kv_status i8kv_bf16_paged_decode_attn(void* out, int out_dtype, const uint16_t* q, const uint16_t* k_cache,
                                        const uint16_t* v_cache, const int32_t* block_tables,
                                        const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int block_size,
                                        int max_blocks, int num_blocks, float softmax_scale, int partition,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  i8kv::DecodeParams p{};
  i8kv_status s = decode_common(p, q, nullptr, false, k_cache, v_cache, nullptr, nullptr, block_tables, seq_lens, B,
                                Hq, Hkv, D, block_size, max_blocks, num_blocks, softmax_scale, partition, workspace,
                                workspace_bytes, out, out_dtype);
  if (s != I8KV_OK || B == 0) return s;
  return from_cuda(i8kv::launch_bf16_decode(p, static_cast<cudaStream_t>(stream)), "bf16 decode launch");
}

}  // extern "C"
