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
//
// The fused variant ([KV] §2.2 step 2, §5.3) first applies a per-head RMSNorm
// and rotate-half RoPE to each Q and K vector in fp32, every operation a single
// correctly rounded one in a fixed order, so its cache bytes are reproducible
// too.  The tile's 16 rows of the cos/sin table are staged in shared memory
// once; a lane's rotation partner (head dim i +- rd/2) sits rd/32 lanes away in
// the same lane group and is fetched by shuffle.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace i8kv {

namespace {

constexpr int kTileTokens = 16;
constexpr int kMaxHkvProducer = 8;

// Quantize the vector whose 16-element slice this lane holds (lane c of a group
// of LPV lanes holds elements 16c .. 16c+15 in x; an inactive lane holds zeros).
// Every lane of the warp must call this (the absmax reduction shuffles across
// the whole warp).  Returns the vector's scale; writes this lane's 16 codes.
template <int LPV>
__device__ __forceinline__ float quantize_slice(const float (&x)[16], uint4& codes) {
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
  uint32_t q[16];
  if (amax > 0.f) {
    div_rne_row(x, scale, __frcp_rn(scale), q);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = 0;
  }
  uint32_t pk[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    pk[j] = __byte_perm(__byte_perm(q[4 * j], q[4 * j + 1], 0x0040), __byte_perm(q[4 * j + 2], q[4 * j + 3], 0x0040),
                        0x5410);
  codes = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  return amax > 0.f ? scale : 0.f;
}

__device__ __forceinline__ void bf16x16_to_f32(const uint4 (&raw)[2], bool active, float (&x)[16]) {
  const uint32_t w[8] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w, raw[1].x, raw[1].y, raw[1].z, raw[1].w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = active ? bf16_bits_to_float(w[i] & 0xffffu) : 0.f;
    x[2 * i + 1] = active ? bf16_bits_to_float(w[i] >> 16) : 0.f;
  }
}

// RMSNorm then rotate-half RoPE of one Q or K head vector, each step a single
// correctly rounded fp32 operation (explicit _rn intrinsics: nothing may be
// contracted into an FMA), in this order:
//   ss   = sum of x_i^2 as a balanced binary tree in index order (the lane's
//          16 elements, then the lane group by xor-shuffles 1, 2, 4, ...;
//          fp32 addition is commutative, so both lanes of a pair get one value)
//   inv  = 1 / sqrt(ss * (1/D) + eps);   y_i = (x_i * inv) * w_i
//   RoPE on the first rd dims, h = rd/2, row cs = (cos_0..cos_{h-1}, sin_0..):
//   y_i = a c_i - b s_i,  y_{i+h} = b c_i + a s_i  (a = y_i, b = y_{i+h}).
// Source: [KV] §2.2 (RoPE on Q/K inside the producer, before the absmax) and
// §5.3 (the per-head Q/K RMSNorm ahead of RoPE).  Every lane of the warp calls
// this (shuffles); `norm` / `rope` select what applies to this lane's vector.
// hc = rd / 32 is the lane distance between a pair's two elements.
template <int LPV>
__device__ __forceinline__ void norm_rope_slice(float (&x)[16], int lane, int c, bool norm, const float* w16,
                                                float eps, bool rope, int hc, int h, const float* cs) {
  if (__any_sync(0xffffffffu, norm)) {
    float s8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint64_t v = f2(x[2 * i], x[2 * i + 1]);
      float lo, hi;
      f2_split(mul2(v, v), lo, hi);
      s8[i] = __fadd_rn(lo, hi);
    }
#pragma unroll
    for (int n = 4; n >= 1; n >>= 1)
#pragma unroll
      for (int i = 0; i < n; ++i) s8[i] = __fadd_rn(s8[2 * i], s8[2 * i + 1]);
    float ss = s8[0];
#pragma unroll
    for (int o = 1; o < LPV; o <<= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    if (norm) {
      const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(ss, 1.0f / (16 * LPV)), eps)));
      const uint64_t inv2 = f2(inv, inv);
#pragma unroll
      for (int j4 = 0; j4 < 4; ++j4) {
        const float4 w = *reinterpret_cast<const float4*>(w16 + 4 * j4);
        f2_split(mul2(mul2(f2(x[4 * j4], x[4 * j4 + 1]), inv2), f2(w.x, w.y)), x[4 * j4], x[4 * j4 + 1]);
        f2_split(mul2(mul2(f2(x[4 * j4 + 2], x[4 * j4 + 3]), inv2), f2(w.z, w.w)), x[4 * j4 + 2], x[4 * j4 + 3]);
      }
    }
  }
  // Partner lane: c <-> c + hc for c < 2 hc.  A shuffle samples every lane's
  // x[j] before any lane overwrites it, so the update follows each exchange.
  // The first-half lane needs a c - b s: it adds b * (-s), negation being
  // exact, so both halves run the same multiply-multiply-add.
  const bool first = c < hc;
  const bool rot = rope && c < 2 * hc;
  if (__any_sync(0xffffffffu, rot)) {
    const int src = rot ? (first ? lane + hc : lane - hc) : lane;
    const int i0 = rot ? 16 * (first ? c : c - hc) : 0;
    const uint32_t neg = first ? 0x80000000u : 0u;
#pragma unroll
    for (int j4 = 0; j4 < 4; ++j4) {
      const float4 cv = *reinterpret_cast<const float4*>(cs + i0 + 4 * j4);
      const float4 sv = *reinterpret_cast<const float4*>(cs + h + i0 + 4 * j4);
      const float sn[4] = {__uint_as_float(__float_as_uint(sv.x) ^ neg), __uint_as_float(__float_as_uint(sv.y) ^ neg),
                           __uint_as_float(__float_as_uint(sv.z) ^ neg), __uint_as_float(__float_as_uint(sv.w) ^ neg)};
      float o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = __shfl_sync(0xffffffffu, x[4 * j4 + e], src);
      // Packed products, scalar sums: ptxas contracts a packed add fed by a
      // packed multiply into a fused multiply-add, which would skip the
      // product's rounding; a scalar add of the halves keeps both roundings.
      float a[4], b[4];
      f2_split(mul2(f2(x[4 * j4], x[4 * j4 + 1]), f2(cv.x, cv.y)), a[0], a[1]);
      f2_split(mul2(f2(x[4 * j4 + 2], x[4 * j4 + 3]), f2(cv.z, cv.w)), a[2], a[3]);
      f2_split(mul2(f2(o[0], o[1]), f2(sn[0], sn[1])), b[0], b[1]);
      f2_split(mul2(f2(o[2], o[3]), f2(sn[2], sn[3])), b[2], b[3]);
#pragma unroll
      for (int e = 0; e < 4; ++e) x[4 * j4 + e] = rot ? __fadd_rn(a[e], b[e]) : x[4 * j4 + e];
    }
  }
}

__device__ __forceinline__ void store_bf16x16(uint16_t* dst, const float (&x)[16]) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x[2 * i])) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x[2 * i + 1])) << 16);
  *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(dst + 8) = make_uint4(w[4], w[5], w[6], w[7]);
}

// kFused adds the RMSNorm / RoPE step on Q and K (and the optional bf16 copies
// of the transformed vectors) and the optional per-channel K smoothing (K times
// RN(1/s), Q times s of its KV head); it then takes its shared memory
// dynamically: [16 tokens][rd] fp32 table rows, the smoothing factors [Hkv][D]
// and their reciprocals [Hkv][D] (when given), then the V staging tile [Hkv][16][D].
template <int D, bool kFused>
__global__ void __launch_bounds__(256, 4) kv_quant_write_kernel(ProducerParams p) {
  constexpr int LPV = D / 16;    // lanes per vector
  constexpr int VPW = 32 / LPV;  // vectors per warp pass
  constexpr int BS = 16;
  __shared__ __align__(16) int8_t vstage_s[kFused ? 16 : kMaxHkvProducer * kTileTokens * D];
  __shared__ int s_slot[kTileTokens];
  __shared__ int s_pos[kTileTokens];                        // fused: table row; -1 = token skipped
  __shared__ __align__(16) float s_w[2][kFused ? D : 4];  // fused: Q, K norm weights (fp32)
  extern __shared__ __align__(16) uint8_t dsm[];
  const int rd = kFused ? p.rd : 0;
  const bool smooth = kFused && p.k_smooth != nullptr;
  const float* s_cs = reinterpret_cast<const float*>(dsm);
  float* s_sm = reinterpret_cast<float*>(dsm + (size_t)kTileTokens * rd * sizeof(float));  // s, then RN(1/s)
  const size_t sm_bytes = smooth ? (size_t)2 * p.Hkv * D * sizeof(float) : 0;
  int8_t* vstage = kFused ? reinterpret_cast<int8_t*>(dsm + (size_t)kTileTokens * rd * sizeof(float) + sm_bytes)
                          : vstage_s;

  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kTileTokens;
  const int ntok = min(kTileTokens, p.T - t0);
  const long long pool_slots = (long long)p.num_blocks * BS;
  if (tid < kTileTokens) {
    int s = -1, pos = -1;
    if (tid < ntok) {
      s = p.slots[t0 + tid];
      if (s >= pool_slots) {
        record_error(2);
        s = -1;
      }
      pos = 0;
      if (kFused && rd > 0) {
        pos = p.positions[t0 + tid];
        if (pos < 0 || pos >= p.max_pos) {  // outside the table: the token is skipped
          record_error(4);
          pos = -1;
          s = -1;
        }
      }
    }
    s_slot[tid] = s;
    s_pos[tid] = pos;
  }
  if constexpr (kFused) {
    for (int i = tid; i < 2 * D; i += blockDim.x) {
      const uint16_t* w = i < D ? p.q_norm_w : p.k_norm_w;
      if (w) s_w[i / D][i % D] = bf16_bits_to_float(__ldg(w + i % D));
    }
    if (smooth) {
      for (int i = tid; i < p.Hkv * D; i += blockDim.x) {
        const float f = __ldg(p.k_smooth + i);
        s_sm[i] = f;
        s_sm[p.Hkv * D + i] = __frcp_rn(f);
      }
    }
    if (rd > 0) {
      __syncthreads();  // s_pos
      const int r4 = rd / 4;
      for (int i = tid; i < kTileTokens * r4; i += blockDim.x) {
        const int tok = i / r4, j = i - tok * r4;
        const int pos = s_pos[tok];
        if (pos >= 0)
          reinterpret_cast<float4*>(dsm)[i] = __ldg(reinterpret_cast<const float4*>(p.cos_sin + (size_t)pos * rd) + j);
      }
    }
  }
  __syncthreads();
  // The tile fills exactly one block, in order: V goes out transposed.
  bool aligned = (ntok == kTileTokens) && s_slot[0] >= 0 && (s_slot[0] % BS) == 0;
#pragma unroll
  for (int i = 1; i < kTileTokens; ++i) aligned = aligned && (s_slot[i] == s_slot[0] + i);

  const int Hkv = p.Hkv, Hq = p.q ? p.Hq : 0;
  const bool k_copy = kFused && p.k_out != nullptr;
  const int hc = rd / 32, hrd = rd / 2;
  // Only the tile's real tokens: vector vi is (token vi / per_tok, entry vi % per_tok),
  // entries 0..Hkv-1 = K heads, Hkv..2Hkv-1 = V heads, then the query heads.
  const int per_tok = 2 * Hkv + Hq;
  const int nvec = ntok * per_tok;
  const int gi = lane / LPV, c = lane % LPV;
  // U warp passes at a time: their loads are issued before either is used, so
  // two global-load latencies overlap instead of queuing one per pass (the
  // fused variant's transform needs the registers: one pass at a time).
  constexpr int U = kFused ? 1 : 2;
  for (int base0 = warp * VPW; base0 < nvec; base0 += 8 * VPW * U) {
    // Per pass: meta = tok | kind << 5 | h << 8 | active << 31, and the slot.
    uint32_t meta[U];
    int slots[U];
    uint4 raw[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = base0 + u * 8 * VPW + gi;
      const int tok = vi / per_tok, r = vi % per_tok;
      const int kind = r < Hkv ? 0 : (r < 2 * Hkv ? 1 : 2);  // 0 = K, 1 = V, 2 = Q
      const int h = kind == 0 ? r : (kind == 1 ? r - Hkv : r - 2 * Hkv);
      bool active = vi < nvec;
      const int slot = active ? s_slot[tok] : -1;
      if (kFused) active = active && s_pos[tok] >= 0;
      if (kind == 1 || (kind == 0 && !k_copy)) active = active && slot >= 0;
      meta[u] = (uint32_t)min(tok, kTileTokens - 1) | ((uint32_t)kind << 5) | ((uint32_t)h << 8) |
                (active ? 0x80000000u : 0u);
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
      const bool act = (meta[u] >> 31) != 0;
      const int tok = meta[u] & 31, kind = (meta[u] >> 5) & 3, h = (meta[u] >> 8) & 0x7fffff;
      float x[16];
      bf16x16_to_f32(raw[u], act, x);
      const int t = t0 + tok;
      if constexpr (kFused) {
        const bool norm = act && ((kind == 0 && p.k_norm_w) || (kind == 2 && p.q_norm_w));
        norm_rope_slice<LPV>(x, lane, c, norm, &s_w[kind == 0 ? 1 : 0][16 * c], p.eps, act && kind != 1 && rd > 0,
                             hc, hrd, s_cs + (size_t)tok * rd);
        if (act) {
          if (kind == 0 && p.k_out) store_bf16x16(p.k_out + ((size_t)t * Hkv + h) * D + 16 * c, x);
          if (kind == 2 && p.q_out) store_bf16x16(p.q_out + ((size_t)t * Hq + h) * D + 16 * c, x);
          if (smooth && kind != 1) {
            // K: times RN(1/s[h]); Q: times s[h / G]
            const float* f = s_sm + (kind == 0 ? (size_t)Hkv * D + (size_t)h * D : (size_t)(h / (Hq / Hkv)) * D) +
                             16 * c;
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              const float4 m = *reinterpret_cast<const float4*>(f + 4 * j4);
              f2_split(mul2(f2(x[4 * j4], x[4 * j4 + 1]), f2(m.x, m.y)), x[4 * j4], x[4 * j4 + 1]);
              f2_split(mul2(f2(x[4 * j4 + 2], x[4 * j4 + 3]), f2(m.z, m.w)), x[4 * j4 + 2], x[4 * j4 + 3]);
            }
          }
        }
      }
      uint4 codes;
      const float scale = quantize_slice<LPV>(x, codes);
      if (!act) continue;
      if (kind == 2) {
        if (kFused && !p.q_i8) continue;
        *reinterpret_cast<uint4*>(p.q_i8 + ((size_t)t * Hq + h) * D + 16 * c) = codes;
        if (c == 0) p.q_scale[(size_t)t * Hq + h] = scale;
        continue;
      }
      const int slot = slots[u];
      if (slot < 0) continue;  // K copied to k_out only
      const int blk = slot / BS, off = slot % BS;
      const size_t sidx = ((size_t)blk * BS + off) * Hkv + h;
      if (kind == 0) {
        *reinterpret_cast<uint4*>(p.k_cache + ((((size_t)blk * Hkv + h) * (D / 16) + c) * BS + off) * 16) = codes;
        if (c == 0) p.k_scale[sidx] = scale;
      } else {
        if (aligned) {
          *reinterpret_cast<uint4*>(&vstage[((size_t)h * kTileTokens + tok) * D + 16 * c]) = codes;
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
      for (int i = 0; i < 4; ++i)
        w[i] = *reinterpret_cast<const uint32_t*>(&vstage[((size_t)h * kTileTokens + 4 * t4 + i) * D + 4 * d4]);
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
  if (p.D == 256) return launch_pdl(kv_quant_write_kernel<256, false>, dim3(grid), dim3(256), 0, stream, p);
  return launch_pdl(kv_quant_write_kernel<128, false>, dim3(grid), dim3(256), 0, stream, p);
}

// Dynamic shared memory: the tile's table rows, then the V staging tile.
static size_t fused_smem_bytes(const ProducerParams& p) {
  return (size_t)kTileTokens * p.rd * sizeof(float) + (p.k_smooth ? (size_t)2 * p.Hkv * p.D * sizeof(float) : 0) +
         (size_t)p.Hkv * kTileTokens * p.D;
}

cudaError_t launch_kv_rope_quant_write(const ProducerParams& p, cudaStream_t stream) {
  const int grid = (p.T + kTileTokens - 1) / kTileTokens;
  if (grid == 0) return cudaSuccess;
  const size_t smem = fused_smem_bytes(p);
  // At most 16 x 256 x 4 + 2 x 8 x 256 x 4 + 8 x 16 x 256 = 64 KB; allow it past the default cap.
  constexpr int kMaxDyn = kTileTokens * 256 * 4 + 2 * kMaxHkvProducer * 256 * 4 + kMaxHkvProducer * kTileTokens * 256;
  auto kernel = p.D == 256 ? kv_quant_write_kernel<256, true> : kv_quant_write_kernel<128, true>;
  // the shared-memory opt-in, once per (device, head_dim); setting it twice is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  static bool opted_in[64][2] = {};
  const bool track = dev >= 0 && dev < 64;
  if (!track || !opted_in[dev][p.D == 256 ? 1 : 0]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDyn);
    if (e != cudaSuccess) return e;
    if (track) opted_in[dev][p.D == 256 ? 1 : 0] = true;
  }
  return launch_pdl(kernel, dim3(grid), dim3(256), smem, stream, p);
}

cudaError_t launch_bf16_kv_write(const ProducerParams& p, uint16_t* k_cache, uint16_t* v_cache, cudaStream_t stream) {
  const long long total = (long long)p.T * p.Hkv * (p.D / 8);
  if (total == 0) return cudaSuccess;
  const int grid = (int)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
  bf16_kv_write_kernel<<<grid, 256, 0, stream>>>(p, k_cache, v_cache);
  return cudaGetLastError();
}

}  // namespace i8kv
