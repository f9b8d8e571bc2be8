// producer.cu -- the fused KV producer: per-(token, head) absmax INT8
// quantization of K, V (and optionally Q) and the scatter into the paged cache.
//
// Source: "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化", §2.1 (the
// quantization rule), §2.2 (the fused producer: absmax, scale, quantize, paged
// write and scale write in one kernel, query quantized once) and §2.3 (layouts).
//
// GB300 shape.  A CTA owns a tile of 16 consecutive tokens.  Each (token, head)
// vector is held by a group of D/16 lanes, 16 bf16 per lane (two 16-byte loads);
// the absmax is a shuffle reduction inside the lane group.  K and Q codes leave
// as one 16-byte store per lane (K's 16-dim chunk layout makes a lane's codes
// contiguous).  V is token-inner: when the tile's 16 tokens fill one whole
// block (the common prefill case) the codes are staged in shared memory and
// written transposed, 4 bytes per store; otherwise each lane writes its 16
// codes byte by byte.
//
// Bit-exactness: scale = amax / 127 and x / scale are IEEE fp32 divisions,
// codes are round-half-to-even; the build does not use fast-math.
#include "common.cuh"
#include "kernels.h"

namespace i8kv {

namespace {

constexpr int kTileTokens = 16;
constexpr int kMaxHkvProducer = 8;

// Quantize the vector whose 16-element slice this lane holds (lane c of a group
// of LPV lanes holds elements 16c .. 16c+15, as raw bf16 words in `raw`).
// Every lane of the warp must call this (the absmax reduction shuffles across
// the whole warp).  Returns the vector's scale; writes this lane's 16 codes.
template <int LPV>
__device__ __forceinline__ float quantize_slice(const uint4 (&raw)[2], bool active, uint4& codes) {
  float x[16];
  const uint32_t w[8] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w, raw[1].x, raw[1].y, raw[1].z, raw[1].w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = active ? bf16_bits_to_float(w[i] & 0xffffu) : 0.f;
    x[2 * i + 1] = active ? bf16_bits_to_float(w[i] >> 16) : 0.f;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = LPV / 2; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = div127(amax);  // amax / 127, correctly rounded
  // Codes: round half to even by adding 1.5 * 2^23 (the fp32 sum keeps the
  // integer part of x / scale in its low mantissa bits, so its low byte is the
  // two's-complement code).  |x / scale| <= amax / RN(amax / 127) < 127.5, so no
  // code ever needs clamping to [-127, 127].
  if (amax > 0.f) {
    div_row(x, scale, __frcp_rn(scale));
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = 0.f;
  }
  uint32_t q[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) q[i] = rne_bits(x[i]);
  uint32_t pk[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    pk[j] = __byte_perm(__byte_perm(q[4 * j], q[4 * j + 1], 0x0040), __byte_perm(q[4 * j + 2], q[4 * j + 3], 0x0040),
                        0x5410);
  codes = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  return amax > 0.f ? scale : 0.f;
}

template <int D>
__global__ void __launch_bounds__(256) kv_quant_write_kernel(ProducerParams p) {
  constexpr int LPV = D / 16;    // lanes per vector
  constexpr int VPW = 32 / LPV;  // vectors per warp pass
  constexpr int BS = 16;
  __shared__ __align__(16) int8_t vstage[kMaxHkvProducer][kTileTokens][D];
  __shared__ int s_slot[kTileTokens];

  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kTileTokens;
  const int ntok = min(kTileTokens, p.T - t0);
  const long long pool_slots = (long long)p.num_blocks * BS;
  if (tid < kTileTokens) {
    int s = -1;
    if (tid < ntok) {
      s = p.slots[t0 + tid];
      if (s >= pool_slots) {
        record_error(2);
        s = -1;
      }
    }
    s_slot[tid] = s;
  }
  __syncthreads();
  // The tile fills exactly one block, in order: V goes out transposed.
  bool aligned = (ntok == kTileTokens) && s_slot[0] >= 0 && (s_slot[0] % BS) == 0;
#pragma unroll
  for (int i = 1; i < kTileTokens; ++i) aligned = aligned && (s_slot[i] == s_slot[0] + i);

  const int Hkv = p.Hkv, Hq = p.q ? p.Hq : 0;
  // Only the tile's real tokens: vector vi is (token vi / per_tok, entry vi % per_tok),
  // entries 0..Hkv-1 = K heads, Hkv..2Hkv-1 = V heads, then the query heads.
  const int per_tok = 2 * Hkv + Hq;
  const int nvec = ntok * per_tok;
  const int gi = lane / LPV, c = lane % LPV;
  // U warp passes at a time: their loads are issued before either is used, so
  // two global-load latencies overlap instead of queuing one per pass.
  constexpr int U = 2;
  for (int base0 = warp * VPW; base0 < nvec; base0 += 8 * VPW * U) {
    bool act[U];
    int kinds[U], toks[U], hs[U], slots[U];
    uint4 raw[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = base0 + u * 8 * VPW + gi;
      const int tok = vi / per_tok, r = vi % per_tok;
      const int kind = r < Hkv ? 0 : (r < 2 * Hkv ? 1 : 2);  // 0 = K, 1 = V, 2 = Q
      const int h = kind == 0 ? r : (kind == 1 ? r - Hkv : r - 2 * Hkv);
      bool active = vi < nvec;
      const int slot = active ? s_slot[tok] : -1;
      if (kind != 2) active = active && slot >= 0;
      act[u] = active;
      kinds[u] = kind;
      toks[u] = tok;
      hs[u] = h;
      slots[u] = slot;
      raw[u][0] = raw[u][1] = make_uint4(0, 0, 0, 0);
      if (active) {
        const int t = t0 + tok;
        const uint16_t* src = (kind == 0 ? p.k + ((size_t)t * Hkv + h) * D
                               : kind == 1 ? p.v + ((size_t)t * Hkv + h) * D
                                           : p.q + ((size_t)t * Hq + h) * D) + 16 * c;
        raw[u][0] = __ldg(reinterpret_cast<const uint4*>(src));
        raw[u][1] = __ldg(reinterpret_cast<const uint4*>(src + 8));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      uint4 codes;
      const float scale = quantize_slice<LPV>(raw[u], act[u], codes);
      if (!act[u]) continue;
      const int kind = kinds[u], tok = toks[u], h = hs[u], slot = slots[u];
      const int t = t0 + tok;
      if (kind == 2) {
        *reinterpret_cast<uint4*>(p.q_i8 + ((size_t)t * Hq + h) * D + 16 * c) = codes;
        if (c == 0) p.q_scale[(size_t)t * Hq + h] = scale;
        continue;
      }
      const int blk = slot / BS, off = slot % BS;
      const size_t sidx = ((size_t)blk * BS + off) * Hkv + h;
      if (kind == 0) {
        *reinterpret_cast<uint4*>(p.k_cache + ((((size_t)blk * Hkv + h) * (D / 16) + c) * BS + off) * 16) = codes;
        if (c == 0) p.k_scale[sidx] = scale;
      } else {
        if (aligned) {
          *reinterpret_cast<uint4*>(&vstage[h][tok][16 * c]) = codes;
        } else {
          int8_t* dst = p.v_cache + (((size_t)blk * Hkv + h) * D + 16 * c) * BS + off;
          const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
          for (int i = 0; i < 16; ++i) dst[(size_t)i * BS] = (int8_t)((w[i >> 2] >> (8 * (i & 3))) & 0xff);
        }
        if (c == 0) p.v_scale[sidx] = scale;
      }
    }
  }
  if (aligned) {
    __syncthreads();
    // 4 tokens x 4 dims per task: read 4 words (token rows), transpose the 4x4
    // byte tile with byte permutes, write 4 words (dim rows, token-inner).
    const int blk = s_slot[0] / BS;
    const int ntask = Hkv * (D / 4) * 4;
    for (int task = tid; task < ntask; task += blockDim.x) {
      const int t4 = task & 3;
      const int d4 = (task >> 2) % (D / 4);
      const int h = (task >> 2) / (D / 4);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = *reinterpret_cast<const uint32_t*>(&vstage[h][4 * t4 + i][4 * d4]);
      const uint32_t x0 = __byte_perm(w[0], w[1], 0x5140), x1 = __byte_perm(w[0], w[1], 0x7362);
      const uint32_t y0 = __byte_perm(w[2], w[3], 0x5140), y1 = __byte_perm(w[2], w[3], 0x7362);
      const uint32_t o[4] = {__byte_perm(x0, y0, 0x5410), __byte_perm(x0, y0, 0x7632), __byte_perm(x1, y1, 0x5410),
                             __byte_perm(x1, y1, 0x7632)};
      int8_t* dst = p.v_cache + (((size_t)blk * Hkv + h) * D + 4 * d4) * BS + 4 * t4;
#pragma unroll
      for (int j = 0; j < 4; ++j) *reinterpret_cast<uint32_t*>(dst + (size_t)j * BS) = o[j];
    }
  }
}

// BF16 comparison cache: K [NB, Hkv, D/8, bs, 8], V [NB, Hkv, D, bs].
// One thread per (token, head, 8-dim chunk).
__global__ void __launch_bounds__(256) bf16_kv_write_kernel(ProducerParams p, uint16_t* kc, uint16_t* vc) {
  constexpr int BS = 16;
  const int D = p.D, Hkv = p.Hkv;
  const long long total = (long long)p.T * Hkv * (D / 8);
  const long long pool_slots = (long long)p.num_blocks * BS;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(i % (D / 8));
    const int h = (int)((i / (D / 8)) % Hkv);
    const int t = (int)(i / ((long long)(D / 8) * Hkv));
    const int slot = p.slots[t];
    if (slot < 0) continue;
    if (slot >= pool_slots) {
      record_error(2);
      continue;
    }
    const int blk = slot / BS, off = slot % BS;
    const uint4 kk = __ldg(reinterpret_cast<const uint4*>(p.k + ((size_t)t * Hkv + h) * D + 8 * c));
    *reinterpret_cast<uint4*>(kc + ((((size_t)blk * Hkv + h) * (D / 8) + c) * BS + off) * 8) = kk;
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(p.v + ((size_t)t * Hkv + h) * D + 8 * c));
    const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
    uint16_t* dst = vc + (((size_t)blk * Hkv + h) * D + 8 * c) * BS + off;
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[(size_t)j * BS] = (uint16_t)((w[j >> 1] >> (16 * (j & 1))) & 0xffffu);
  }
}

}  // namespace

I8KV_DEFINE_ERROR_ACCESSOR(read_error_producer)

cudaError_t launch_kv_quant_write(const ProducerParams& p, cudaStream_t stream) {
  const int grid = (p.T + kTileTokens - 1) / kTileTokens;
  if (grid == 0) return cudaSuccess;
  if (p.D == 256) return launch_pdl(kv_quant_write_kernel<256>, dim3(grid), dim3(256), 0, stream, p);
  return launch_pdl(kv_quant_write_kernel<128>, dim3(grid), dim3(256), 0, stream, p);
}

cudaError_t launch_bf16_kv_write(const ProducerParams& p, uint16_t* k_cache, uint16_t* v_cache, cudaStream_t stream) {
  const long long total = (long long)p.T * p.Hkv * (p.D / 8);
  if (total == 0) return cudaSuccess;
  const int grid = (int)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
  bf16_kv_write_kernel<<<grid, 256, 0, stream>>>(p, k_cache, v_cache);
  return cudaGetLastError();
}

}  // namespace i8kv
