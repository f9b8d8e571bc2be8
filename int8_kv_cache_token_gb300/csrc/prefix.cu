// prefix.cu -- INT8 prefix-prefill chunk attention on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory).
//
// Source: "gfx936 DCU上实现INT8 PV MMAC：V Scale融合、概率量化与Fragment分组"
// §2.1 (the prefix keeps one online softmax (m, l, o); alpha = exp(m - m'),
// p~ = exp(score - m'), W = p~ x sV is quantized unnormalized; O = o / l at
// the end), §1 and §3 (32-token probability groups, sW = max W / 127, W on the
// A side and V on the B side of the INT8 MMA) and "gfx936 DCU上实现INT8 KV与
// INT8 MMAC Attention推理优化" §3.2 (history and the chunk's own K/V in one
// online softmax, never two attentions merged afterwards).
//
// GB300 shape.  A CTA owns 128 query rows of one KV head -- (chunk token, query
// head) pairs of that head's GQA group, token-major, so the query heads sharing
// K/V read the same tiles -- and walks the keys in 32-key probability groups:
//   S  = Qq x Kq^T        tcgen05, M = 128, N = 32, K = D, into TMEM
//   scores, causal mask, p~ = exp(s - m_g) against the group's own row
//   maximum m_g, W = p~ sV, sW = max W / 127, Wq = round(W / sW)
//                         CUDA cores, one thread per row
//   PV = Wq x Vq          tcgen05, M = 128, N = D, K = 32, into TMEM
//   o  = alpha o + exp(m_g - m') sW PV,  l = alpha l + exp(m_g - m') l_g
//                         CUDA cores, o in registers (half of D per thread)
// with m' = max(m, m_g) and alpha = exp(m - m').  The codes round(W / sW) do
// not change when W is scaled, so quantizing each group against m_g and
// bringing it to the running maximum in the output update is the pages' online
// softmax, reordered; it lets the softmax of a group start before the previous
// group's maximum is known.  Scores are kept in log2 units (the scale folds in
// log2 e) so every exponential is one ex2.
//
// The int8 codes are exact in f16, every product (<= 127^2) is exact and every
// partial sum stays below 2^22, so f16 MMAs with fp32 accumulation give the
// INT8 contractions' exact integer results.
//
// Operand tiles.  Every one of the row blocks of a KV head multiplies the same
// keys, so the int8 -> f16 conversion (exact) is done once per (KV head,
// 32-key group) by prefix_tiles_kernel, into a workspace tile laid out exactly
// as the MMAs read it in shared memory (K-major, 16-byte chunks XOR-swizzled:
// K as [key][dim] in 128-byte rows, V as [dim][key] in 64-byte rows) followed
// by the group's sK and sV.  The attention kernel moves each tile with one
// bulk copy.
//
// Warps of the attention kernel.  Warp 0 lane 0 issues the tiles' bulk copies
// (a ring of four); warp 1 owns the TMEM allocation and its lane 0 issues every
// MMA, each QK or PV as soon as its operands are ready.  Warpgroups 1 and 2
// (warps 4-7, 8-11) take the softmax of the even and the odd groups, thread =
// row, so the two run side by side; both apply every group's product to their
// half of the output dims.
//
// The same kernel, instantiated with kBF, is the high-precision chunk path
// ("gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" §3.1: the first
// prefill chunk keeps a high-precision attention): bf16 Q and operand tiles
// (history keys read back from the INT8 cache as bf16(code x scale), the
// chunk's own keys as given), bf16 MMAs, and p~ handed to the PV MMA as bf16
// with no group quantization.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace i8kv {
I8KV_DEFINE_ERROR_ACCESSOR(read_error_prefix)

namespace {

constexpr int kBS = 16;
constexpr int kRows = 128;       // query rows per CTA: the MMA's M, one TMEM lane each
constexpr int kGroup = 32;       // keys per probability group
constexpr int kPagesPG = kGroup / kBS;
constexpr int kStages = 4;       // operand tiles in flight
constexpr int kThreads = 384;
constexpr int kLoadWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kCompWarp0 = 4;    // warps 4..11
constexpr int kWGThreads = 128;

// One (KV head, group) operand tile, in global memory and in shared memory.
template <int D>
struct Tile {
  static constexpr int kK16 = kGroup * D * 2;           // f16 K, D/64 atoms of [32 keys][128 B] (SW128)
  static constexpr int kV16 = D * kGroup * 2;           // f16 V, [D][64 B] (SW64)
  static constexpr int oK = 0;
  static constexpr int oV = kK16;
  static constexpr int oSk = kK16 + kV16;               // sK[32], then sV[32]
  static constexpr int kBytes = oSk + 2 * kGroup * 4;   // one bulk copy
  static constexpr int kSlot = (kBytes + 1023) / 1024 * 1024;  // shared-memory stride (SW128 needs 1024-byte bases)
};

template <int D>
struct Lay {
  static constexpr int kQ16 = kRows * D * 2;          // f16 Q, D/64 atoms of [128 rows][128 B]
  static constexpr int kP16 = kRows * kGroup * 2;     // f16 Wq, [128][64 B]
  static constexpr int oQ = 0;
  static constexpr int oTile = oQ + kQ16;             // kStages tiles
  static constexpr int oP = oTile + kStages * Tile<D>::kSlot;  // two slots
  static constexpr int oSt = oP + 2 * kP16;           // four slots of m_g[128], sW[128], l_g[128]
  static constexpr int oBar = oSt + 4 * 3 * kRows * 4;
  // tile_full[4], tile_free[4], qk_done[2], s_free[2], p_full[2], pv_done[2], pv_free, st_full[4]
  static constexpr int kBars = kStages + kStages + 2 + 2 + 2 + 2 + 1 + 4;
  static constexpr int oCtl = oBar + kBars * 8;       // TMEM base, abort flag
  static constexpr int kTotal = oCtl + 16;
  // TMEM: S in columns [0, 64) (two slots of 32), PV in [kPVCol, kPVCol + D)
  static constexpr uint32_t kPVCol = D == 256 ? 256 : 128;
  static constexpr uint32_t kTmemCols = D == 256 ? 512 : 256;
};

// Byte offset of 16-byte chunk `chunk16` of row r in a K-major tile with
// SWZ-byte rows, the chunk index XOR-swizzled by the row's place in its
// 8-row (SWZ = 128) or 8-row-pair (SWZ = 64) pattern, as the tensor cores read it.
template <int SWZ>
__device__ __forceinline__ uint32_t swz_chunk(int r, int chunk16) {
  constexpr int mask = SWZ == 128 ? 7 : 3;
  return (uint32_t)(r * SWZ + ((chunk16 ^ ((r * SWZ >> 7) & mask)) << 4));
}

// 16 int8 codes (one 16-byte chunk) -> 16 exact f16 values, natural order.
__device__ __forceinline__ void s8x16_to_f16(const uint4& v, uint4& h0, uint4& h1) {
  s8x4_to_f16(v.x, h0.x, h0.y);
  s8x4_to_f16(v.y, h0.z, h0.w);
  s8x4_to_f16(v.z, h1.x, h1.y);
  s8x4_to_f16(v.w, h1.z, h1.w);
}

// Maximum and sum of 32 values as balanced trees (depth 5 instead of a
// 31-step chain); the sum's order is fixed, so every thread rounds alike.  The
// maximum uses the three-input max (exact, so the grouping does not matter);
// the sum adds pairs of adjacent partial sums with one packed add, the same
// additions in the same order as the scalar tree.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float tree_max(const float (&a)[32]) {
  float t[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) t[i] = max3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
  t[10] = fmaxf(a[30], a[31]);
  const float u0 = max3(t[0], t[1], t[2]), u1 = max3(t[3], t[4], t[5]), u2 = max3(t[6], t[7], t[8]);
  const float u3 = fmaxf(t[9], t[10]);
  return fmaxf(max3(u0, u1, u2), u3);
}
__device__ __forceinline__ float tree_sum(const float (&a)[32]) {
  float t[16];
#pragma unroll
  for (int i = 0; i < 16; i += 2)
    f2_split(add2(f2(a[i], a[i + 1]), f2(a[i + 16], a[i + 17])), t[i], t[i + 1]);
#pragma unroll
  for (int n = 8; n >= 2; n >>= 1)
#pragma unroll
    for (int i = 0; i < n; i += 2) f2_split(add2(f2(t[i], t[i + 1]), f2(t[i + n], t[i + n + 1])), t[i], t[i + 1]);
  return __fadd_rn(t[0], t[1]);
}

// Bounded wait that gives up at once when the CTA has aborted (error 1 after
// the time limit); every thread still runs the same loop and barriers, so no
// thread waits on a barrier another one skipped.
__device__ __forceinline__ void pwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return;
  if (*abort_flag) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
    if (*abort_flag) return;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      record_error(1);
      *abort_flag = 1;
      return;
    }
  }
}

// ---- operand tiles: one CTA per (group, KV head); the int8 pages and scales
// of the group's 32 keys -> the f16 tile (exact codes) and sK, sV.  Keys past
// the sequence (the last group's tail) get zero codes and scales; the
// attention masks them anyway.
template <int D>
__global__ void __launch_bounds__(256) prefix_tiles_kernel(PrefixParams p) {
  using T = Tile<D>;
  griddep_wait();
  griddep_launch_dependents();
  const int g = blockIdx.x, kvh = blockIdx.y, tid = threadIdx.x;
  const int Hkv = p.Hkv;
  const int ngt = gridDim.x;
  const int max_blk = (p.H + p.C + kBS - 1) / kBS;
  uint8_t* tile = p.tiles + ((size_t)kvh * ngt + g) * T::kBytes;
  int blk[kPagesPG];
#pragma unroll
  for (int i = 0; i < kPagesPG; ++i) {
    const int lb = g * kPagesPG + i;
    blk[i] = lb < max_blk ? p.block_table[lb] : -1;
    if (lb < max_blk && (blk[i] < 0 || blk[i] >= p.num_blocks)) {
      if (tid == 0) record_error(2);
      blk[i] = -1;
    }
  }
  // K page [D/16][16 tokens][16 B] -> [key][D] (SW128 atoms): chunk i = (page, dim chunk, token)
  constexpr int KC = kPagesPG * (D / 16) * kBS;
  for (int i = tid; i < KC; i += 256) {
    const int pg = i / ((D / 16) * kBS), rem = i % ((D / 16) * kBS);
    const int dc = rem / kBS, key = pg * kBS + rem % kBS;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (blk[pg] >= 0)
      v = __ldg(reinterpret_cast<const uint4*>(p.k_cache + ((size_t)blk[pg] * Hkv + kvh) * (D * kBS)) + rem);
    uint4 h0, h1;
    s8x16_to_f16(v, h0, h1);
    uint8_t* atom = tile + T::oK + (size_t)(dc / 4) * (kGroup * 128);
    *reinterpret_cast<uint4*>(atom + swz_chunk<128>(key, 2 * (dc % 4))) = h0;
    *reinterpret_cast<uint4*>(atom + swz_chunk<128>(key, 2 * (dc % 4) + 1)) = h1;
  }
  // V page [D][16 tokens] -> [D][32 keys] (SW64): chunk i = (page, dim)
  for (int i = tid; i < kPagesPG * D; i += 256) {
    const int pg = i / D, d = i % D;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (blk[pg] >= 0)
      v = __ldg(reinterpret_cast<const uint4*>(p.v_cache + ((size_t)blk[pg] * Hkv + kvh) * (D * kBS)) + d);
    uint4 h0, h1;
    s8x16_to_f16(v, h0, h1);
    *reinterpret_cast<uint4*>(tile + T::oV + swz_chunk<64>(d, 2 * pg)) = h0;
    *reinterpret_cast<uint4*>(tile + T::oV + swz_chunk<64>(d, 2 * pg + 1)) = h1;
  }
  if (tid < kGroup) {
    const int pg = tid / kBS;
    float sk = 0.f, sv = 0.f;
    if (blk[pg] >= 0) {
      const size_t si = ((size_t)blk[pg] * kBS + tid % kBS) * Hkv + kvh;
      sk = p.k_scale[si];
      sv = p.v_scale[si];
    }
    float* sc = reinterpret_cast<float*>(tile + T::oSk);
    sc[tid] = sk;
    sc[kGroup + tid] = sv;
  }
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}
__device__ __forceinline__ float s8_at(const uint32_t (&w)[4], int e) {
  return (float)(int8_t)((w[e >> 2] >> (8 * (e & 3))) & 0xffu);
}

// ---- bf16 operand tiles for the high-precision variant: one CTA per (group,
// KV head).  A history key (t < H) is read back from the INT8 cache as
// bf16(code x scale); a chunk key comes from the bf16 k_chunk / v_chunk rows
// as it is; keys past the sequence are zero.  Same tile layout as the f16
// tiles (the scale slots are not used).
template <int D>
__global__ void __launch_bounds__(256) prefix_tiles_bf16_kernel(PrefixParams p) {
  using T = Tile<D>;
  __shared__ __align__(16) uint16_t vrows[kGroup][D + 8];  // the group's chunk V rows (padded rows)
  __shared__ float s_sk[kGroup], s_sv[kGroup];
  griddep_wait();
  griddep_launch_dependents();
  const int g = blockIdx.x, kvh = blockIdx.y, tid = threadIdx.x;
  const int Hkv = p.Hkv, H = p.H, C = p.C;
  const int ngt = gridDim.x;
  const int key0 = g * kGroup;
  uint8_t* tile = p.tiles + ((size_t)kvh * ngt + g) * T::kBytes;
  int blk[kPagesPG];
#pragma unroll
  for (int i = 0; i < kPagesPG; ++i) {
    const int lb = g * kPagesPG + i;
    blk[i] = -1;
    if (lb * kBS < H) {
      const int b = p.block_table[lb];
      if (b < 0 || b >= p.num_blocks) {
        if (tid == 0) record_error(2);
      } else {
        blk[i] = b;
      }
    }
  }
  if (tid < kGroup) {
    const int t = key0 + tid, pg = tid / kBS;
    float sk = 0.f, sv = 0.f;
    if (t < H && blk[pg] >= 0) {
      const size_t si = ((size_t)blk[pg] * kBS + t % kBS) * Hkv + kvh;
      sk = p.k_scale[si];
      sv = p.v_scale[si];
    }
    s_sk[tid] = sk;
    s_sv[tid] = sv;
  }
  for (int i = tid; i < kGroup * (D / 8); i += 256) {
    const int key = i / (D / 8), c8 = i % (D / 8), t = key0 + key;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (t >= H && t < H + C)
      v = __ldg(reinterpret_cast<const uint4*>(p.v_chunk + ((size_t)(t - H) * Hkv + kvh) * D) + c8);
    *reinterpret_cast<uint4*>(&vrows[key][8 * c8]) = v;
  }
  __syncthreads();
  // K: (key, 16-dim chunk) -> [key][D] (SW128 atoms)
  for (int i = tid; i < kGroup * (D / 16); i += 256) {
    const int key = i / (D / 16), dc = i % (D / 16), t = key0 + key;
    uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
    if (t < H) {
      const int pg = key / kBS;
      if (blk[pg] >= 0) {
        const uint4 c = __ldg(reinterpret_cast<const uint4*>(p.k_cache + ((size_t)blk[pg] * Hkv + kvh) * (D * kBS)) +
                              dc * kBS + t % kBS);
        const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
        const float sk = s_sk[key];
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = bf16x2_bits(__fmul_rn(s8_at(cw, 2 * e), sk), __fmul_rn(s8_at(cw, 2 * e + 1), sk));
        h0 = make_uint4(w[0], w[1], w[2], w[3]);
        h1 = make_uint4(w[4], w[5], w[6], w[7]);
      }
    } else if (t < H + C) {
      const uint4* src = reinterpret_cast<const uint4*>(p.k_chunk + ((size_t)(t - H) * Hkv + kvh) * D + 16 * dc);
      h0 = __ldg(src);
      h1 = __ldg(src + 1);
    }
    uint8_t* atom = tile + T::oK + (size_t)(dc / 4) * (kGroup * 128);
    *reinterpret_cast<uint4*>(atom + swz_chunk<128>(key, 2 * (dc % 4))) = h0;
    *reinterpret_cast<uint4*>(atom + swz_chunk<128>(key, 2 * (dc % 4) + 1)) = h1;
  }
  // V: (page, dim) -> 16 keys of [D][32 keys] (SW64)
  for (int i = tid; i < kPagesPG * D; i += 256) {
    const int pg = i / D, d = i % D;
    uint4 c = make_uint4(0, 0, 0, 0);
    if (blk[pg] >= 0) c = __ldg(reinterpret_cast<const uint4*>(p.v_cache + ((size_t)blk[pg] * Hkv + kvh) * (D * kBS)) + d);
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    uint32_t w[8];
#pragma unroll
    for (int e2 = 0; e2 < 8; ++e2) {
      uint32_t half[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = 2 * e2 + u, key = pg * kBS + e;
        half[u] = key0 + key < H ? bf16x2_bits(__fmul_rn(s8_at(cw, e), s_sv[key]), 0.f) & 0xffffu : vrows[key][d];
      }
      w[e2] = half[0] | (half[1] << 16);
    }
    *reinterpret_cast<uint4*>(tile + T::oV + swz_chunk<64>(d, 2 * pg)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(tile + T::oV + swz_chunk<64>(d, 2 * pg + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// kBF: the high-precision variant -- bf16 query and tiles, no scales, and
// the probabilities go to the PV MMA as bf16 p~ (no group quantization).
// kDbg (INT8 only): the same kernel that also records its raw integer
// contractions -- S = Qq x Kq^T as read from TMEM, the codes Wq and each
// group's Wq x Vq as read from TMEM -- for the debug entry point.
template <int D, bool kBF, bool kDbg = false>
__global__ void __launch_bounds__(kThreads, 1) prefix_attn_kernel(PrefixParams p) {
  static_assert(!(kDbg && kBF), "the debug record is for the INT8 path");
  using Ly = Lay<D>;
  using T = Tile<D>;
  constexpr int DH = D / 2;  // output dims per warpgroup
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* tile_full = reinterpret_cast<uint64_t*>(smem + Ly::oBar);  // [g % kStages]: tile g landed
  uint64_t* tile_free = tile_full + kStages;  // [g % kStages]: PV(g) done, the tile slot may be refilled
  uint64_t* qk_done = tile_free + kStages;    // [g & 1]: S(g) in TMEM
  uint64_t* s_free = qk_done + 2;             // [g & 1]: S(g) read
  uint64_t* p_full = s_free + 2;              // [g & 1]: Wq(g) in its slot
  uint64_t* pv_done = p_full + 2;             // [g & 1]: PV(g) in TMEM; the Wq slot free
  uint64_t* pv_free = pv_done + 2;            // PV accumulator read by both warpgroups
  uint64_t* st_full = pv_free + 1;            // [g & 3]: the group's row statistics
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::oCtl);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::oCtl + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G, Hq = p.Hq, H = p.H, C = p.C;
  const int R = C * G;
  // Work item -> (row block, KV head, part).  Row blocks in reverse order, the
  // KV heads interleaved: later chunk tokens see more keys, and CTAs start in
  // index order, so the heaviest blocks run first and the last wave holds the
  // lightest ones -- which are split over their key groups (split_k parts), so
  // that the last wave's work spreads over the SMs instead of leaving them idle.
  int blk = blockIdx.x, part = 0, nparts = 1;
  if (blk >= p.full_items) {
    const int t = blk - p.full_items;
    blk = p.full_items + t / p.split_k;
    part = t % p.split_k;
    nparts = p.split_k;
  }
  const int kvh = blk % p.Hkv;
  const int r0 = (p.nrb - 1 - blk / p.Hkv) * kRows;
  const int j_hi = min(C - 1, (r0 + kRows - 1) / G);
  const int n_keys = H + j_hi + 1;
  const int ng_all = (n_keys + kGroup - 1) / kGroup;
  // this part's key groups [g_begin, g_begin + ng); the pipeline counts from 0
  const int g_begin = (int)((long long)ng_all * part / nparts);
  const int ng = (int)((long long)ng_all * (part + 1) / nparts) - g_begin;
  const int ngt = (H + C + kGroup - 1) / kGroup;  // groups of the whole sequence (tiles per KV head)

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&tile_full[s], 1);
      mbar_init(&tile_free[s], 1);
    }
    for (int s = 0; s < 4; ++s) mbar_init(&st_full[s], kWGThreads);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qk_done[s], 1);
      mbar_init(&s_free[s], kWGThreads);
      mbar_init(&p_full[s], kWGThreads);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(pv_free, 2 * kWGThreads);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, Ly::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // From here on the kernel reads what earlier work on the stream wrote (the
  // query and the operand tiles).
  griddep_wait();
  griddep_launch_dependents();

  // ---- Q tile -> f16 (all threads), K-major SW128 ----
  {
    uint8_t* q16 = smem + Ly::oQ;
    constexpr int CH = D / 16;  // int8 chunks per row
    for (int i = tid; i < kRows * CH; i += kThreads) {
      const int rr = i / CH, dc = i % CH;
      const int r = r0 + rr;
      uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
      if constexpr (kBF) {
        if (r < R) {
          const int j = r / G, hq = kvh * G + r % G;
          const uint4* src = reinterpret_cast<const uint4*>(p.qb + ((size_t)j * Hq + hq) * D) + 2 * dc;
          h0 = __ldg(src);
          h1 = __ldg(src + 1);
        }
      } else {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < R) {
          const int j = r / G, hq = kvh * G + r % G;
          v = __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t)j * Hq + hq) * D) + dc);
        }
        s8x16_to_f16(v, h0, h1);
      }
      uint8_t* atom = q16 + (size_t)(dc / 4) * (kRows * 128);
      *reinterpret_cast<uint4*>(atom + swz_chunk<128>(rr, 2 * (dc % 4))) = h0;
      *reinterpret_cast<uint4*>(atom + swz_chunk<128>(rr, 2 * (dc % 4) + 1)) = h1;
    }
    fence_async_smem();
  }
  __syncthreads();

  if (warp < kCompWarp0) {
    regs_dec<64>();  // warpgroup 0 hands registers to the softmax/output warpgroups
    if (warp == kLoadWarp && lane == 0) {
      // ================= tile copies (warp 0, lane 0) =================
      const uint8_t* src = p.tiles + (size_t)kvh * ngt * T::kBytes;
      int g = 0;
      for (; g < ng; ++g) {
        const int st = g % kStages;
        if (g >= kStages) pwait(&tile_free[st], ((g - kStages) / kStages) & 1, abort_flag);
        if (*abort_flag) break;
        mbar_expect_tx(&tile_full[st], T::kBytes);
        bulk_g2s(smem + Ly::oTile + (size_t)st * T::kSlot, src + (size_t)(g_begin + g) * T::kBytes, T::kBytes,
                 &tile_full[st]);
        mbar_arrive(&tile_full[st]);
      }
      // copies issued but never waited for (after an abort) land before the CTA exits
      for (int k = max(0, g - kStages); k < g; ++k) mbar_wait(&tile_full[k % kStages], (k / kStages) & 1);
    } else if (warp == kMmaWarp && lane == 0) {
      // ================= MMA issue (warp 1, lane 0) =================
      // Whichever of the next QK and the next PV has its operands first is
      // issued; the checks never suspend (test_wait), a pass with nothing to
      // issue sleeps briefly, and the same time limit as pwait applies.
      constexpr uint32_t idesc_qk = kBF ? umma_idesc_bf16(kRows, kGroup) : umma_idesc_f16(kRows, kGroup);
      constexpr uint32_t idesc_pv = kBF ? umma_idesc_bf16(kRows, D) : umma_idesc_f16(kRows, D);
      const uint32_t q16 = smem_u32(smem + Ly::oQ);
      const uint32_t tiles = smem_u32(smem + Ly::oTile);
      int nq = 0, np = 0;  // next QK, next PV
      uint64_t t_idle = 0;
      while (np < ng) {
        bool did = false;
        if (nq < ng && mbar_test(&tile_full[nq % kStages], (nq / kStages) & 1) &&
            (nq < 2 || mbar_test(&s_free[nq & 1], ((nq - 2) >> 1) & 1))) {
          const uint32_t k16 = tiles + (nq % kStages) * T::kSlot + T::oK;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t a = q16 + (kk / 4) * (kRows * 128) + (kk % 4) * 32;
            const uint32_t b = k16 + (kk / 4) * (kGroup * 128) + (kk % 4) * 32;
            umma_f16(tmem + 32 * (nq & 1), umma_desc(a, 128), umma_desc(b, 128), idesc_qk, kk > 0);
          }
          umma_commit(&qk_done[nq & 1]);
          ++nq;
          did = true;
        }
        if (np < nq && mbar_test(&p_full[np & 1], (np >> 1) & 1) &&
            (np < 1 || mbar_test(pv_free, (np - 1) & 1))) {
          const uint32_t p16 = smem_u32(smem + Ly::oP + (size_t)(np & 1) * Ly::kP16);
          const uint32_t v16 = tiles + (np % kStages) * T::kSlot + T::oV;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kGroup / 16; ++kk)
            umma_f16(tmem + Ly::kPVCol, umma_desc(p16 + kk * 32, 64), umma_desc(v16 + kk * 32, 64), idesc_pv,
                     kk > 0);
          umma_commit(&pv_done[np & 1]);
          umma_commit(&tile_free[np % kStages]);
          ++np;
          did = true;
        }
        if (did) {
          t_idle = 0;
        } else {
          if (*abort_flag) break;
          const uint64_t now = global_timer_ns();
          if (t_idle == 0) {
            t_idle = now;
          } else if (now - t_idle > kWaitLimitNs) {
            record_error(1);
            *abort_flag = 1;
            break;
          }
          __nanosleep(32);
        }
      }
      // every MMA issued has completed before TMEM is released (the last commit
      // covers all earlier MMAs)
      if (np >= 1) mbar_wait(&pv_done[(np - 1) & 1], ((np - 1) >> 1) & 1);
      if (nq > np) mbar_wait(&qk_done[(nq - 1) & 1], ((nq - 1) >> 1) & 1);
    }
    __syncwarp();
  } else {
    // ================= softmax and output (warpgroups 1, 2) =================
    regs_inc<216>();
    const int wg = (warp - kCompWarp0) >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int r = r0 + row;
    const bool valid = r < R;
    const int j = valid ? r / G : 0, hq = kvh * G + (valid ? r % G : 0);
    const int lim = valid ? H + j : -1;  // last visible key
    // score in log2 units: acc x sQ x scale x log2(e) x sK
    const float c2 = !valid ? 0.f
                     : kBF  ? __fmul_rn(p.sm_scale, kLog2e)
                            : __fmul_rn(__fmul_rn(p.q_scale[(size_t)j * Hq + hq], p.sm_scale), kLog2e);
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    float* stats = reinterpret_cast<float*>(smem + Ly::oSt);  // [slot][m_g | sW | l_g][row]
    float o[DH];
#pragma unroll
    for (int i = 0; i < DH; ++i) o[i] = 0.f;
    float m = -INFINITY, l = 0.f;

    // softmax of group g (this warpgroup's parity): codes into the Wq slot,
    // (m_g, sW, l_g) into the statistics slot
    auto softmax = [&](int g) {
      const int sl = g & 1;
      pwait(&qk_done[sl], (g >> 1) & 1, abort_flag);
      tc_fence_after();
      float s[32];
      tmem_ld32(trow + 32 * sl, s);
      const int key0 = (g_begin + g) * kGroup;
      const bool full = __all_sync(0xffffffffu, key0 + kGroup - 1 <= lim);  // no key of the warp is masked
      float mg, lg = 0.f, sw = 0.f;
      uint32_t pk[16];
      if constexpr (kBF) {
        tmem_wait_ld();
        {
          const uint64_t cc = f2(c2, c2);
#pragma unroll
          for (int t = 0; t < 16; ++t) f2_split(mul2(f2(s[2 * t], s[2 * t + 1]), cc), s[2 * t], s[2 * t + 1]);
        }
        if (!full) {
#pragma unroll
          for (int t = 0; t < 32; ++t)
            if (key0 + t > lim) s[t] = -INFINITY;
        }
        mg = tree_max(s);
        if (mg != -INFINITY) {
#pragma unroll
          for (int t = 0; t < 32; ++t) s[t] = ex2(__fsub_rn(s[t], mg));  // p~; 0 for a masked key
          lg = tree_sum(s);
          sw = 1.f;
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) s[t] = 0.f;
        }
        tc_fence_before();
        mbar_arrive(&s_free[sl]);  // S is read; QK(g + 2) may overwrite it
        // p~ as bf16, two per register (low half = the even key)
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = bf16x2_bits(s[2 * i], s[2 * i + 1]);
      } else {
      pwait(&tile_full[g % kStages], (g / kStages) & 1, abort_flag);  // the group's scales (already landed)
      const float4* sk4 =
          reinterpret_cast<const float4*>(smem + Ly::oTile + (size_t)(g % kStages) * T::kSlot + T::oSk);
      const float4* sv4 = sk4 + kGroup / 4;
      tmem_wait_ld();
      if constexpr (kDbg) {
        // the raw accumulators of the visible keys (exact integers in fp32)
        if (valid) {
          int32_t* srow = p.dbg_s + ((size_t)j * Hq + hq) * (H + C);
#pragma unroll
          for (int t = 0; t < 32; ++t)
            if (key0 + t <= lim) srow[key0 + t] = __float2int_rn(s[t]);
        }
      }
      {
        const uint64_t cc = f2(c2, c2);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 k4 = sk4[i];
          f2_split(mul2(mul2(f2(s[4 * i], s[4 * i + 1]), f2(k4.x, k4.y)), cc), s[4 * i], s[4 * i + 1]);
          f2_split(mul2(mul2(f2(s[4 * i + 2], s[4 * i + 3]), f2(k4.z, k4.w)), cc), s[4 * i + 2], s[4 * i + 3]);
        }
      }
      if (!full) {
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (key0 + t > lim) s[t] = -INFINITY;
      }
      mg = tree_max(s);
      float A = 0.f;
      if (mg != -INFINITY) {
#pragma unroll
        for (int t = 0; t < 32; ++t) s[t] = ex2(__fsub_rn(s[t], mg));  // p~; 0 for a masked key
        lg = tree_sum(s);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 v4 = sv4[i];
          f2_split(mul2(f2(s[4 * i], s[4 * i + 1]), f2(v4.x, v4.y)), s[4 * i], s[4 * i + 1]);
          f2_split(mul2(f2(s[4 * i + 2], s[4 * i + 3]), f2(v4.z, v4.w)), s[4 * i + 2], s[4 * i + 3]);
        }
        if (!full) {
#pragma unroll
          for (int t = 0; t < 32; ++t)
            if (key0 + t > lim) s[t] = 0.f;
        }
        A = tree_max(s);
      }
      tc_fence_before();
      mbar_arrive(&s_free[sl]);  // S is read; QK(g + 2) may overwrite it
      // sW = A / 127 and the codes round(W / sW), both IEEE fp32 quotients (W / sW
      // by Markstein's method); W / sW <= A / RN(A / 127) < 127.5, no clamp needed
      sw = div127(A);
      if (A > 0.f) {
        // round-half-even(q) + 1024 as the f16 bit pattern 0x6400 + code, from the
        // low bits of the fp32 sum q + 1.5 * 2^23 + 0x6400; two per register, then
        // 1024 subtracted (exact)
        uint32_t qb[32];
        div_rne_row(s, sw, __frcp_rn(sw), qb, 12608512.0f);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t lo = qb[2 * i], hi = qb[2 * i + 1];
          uint32_t h = __byte_perm(lo, hi, 0x5410);
          asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(h) : "r"(0x64006400u));
          pk[i] = h;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = 0u;
      }
      }
      if constexpr (kDbg) {
        if (valid) {
          uint8_t* wrow = p.dbg_wq + ((size_t)j * Hq + hq) * (size_t)(ngt * kGroup);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&pk[i]));
            if (key0 + 2 * i <= lim) wrow[key0 + 2 * i] = (uint8_t)__float2int_rn(c.x);
            if (key0 + 2 * i + 1 <= lim) wrow[key0 + 2 * i + 1] = (uint8_t)__float2int_rn(c.y);
          }
        }
      }
      // Wq (f16) or p~ (bf16) -> the PV A tile, row `row`; then the row statistics
      if (g >= 2) pwait(&pv_done[sl], ((g - 2) >> 1) & 1, abort_flag);  // PV(g-2) has read the slot
      uint8_t* p16 = smem + Ly::oP + (size_t)sl * Ly::kP16;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(p16 + swz_chunk<64>(row, c)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_async_smem();
      mbar_arrive(&p_full[sl]);
      float* st = stats + (g & 3) * 3 * kRows;
      st[row] = mg;
      st[kRows + row] = sw;
      st[2 * kRows + row] = lg;
      mbar_arrive(&st_full[g & 3]);
    };

    // o = alpha o + exp(m_g - m') sW (Wq x Vq), l = alpha l + exp(m_g - m') l_g
    auto update = [&](int h) {
      pwait(&pv_done[h & 1], (h >> 1) & 1, abort_flag);
      pwait(&st_full[h & 3], (h >> 2) & 1, abort_flag);
      const float* st = stats + (h & 3) * 3 * kRows;
      const float mg = st[row], sw = st[kRows + row], lg = st[2 * kRows + row];
      float alpha = 1.f, e = 0.f;
      if (mg != -INFINITY) {
        const float mn = fmaxf(m, mg);
        alpha = m == -INFINITY ? 0.f : ex2(__fsub_rn(m, mn));
        const float f = ex2(__fsub_rn(mg, mn));
        e = __fmul_rn(f, sw);
        l = __fmaf_rn(l, alpha, __fmul_rn(f, lg));
        m = mn;
      }
      tc_fence_after();
      const bool rescale = __any_sync(0xffffffffu, alpha != 1.f);
      // 32-column chunks, two in flight: chunk c + 1 is loading while chunk c
      // joins the output (tcgen05.wait::ld waits for every load issued so far)
      const uint32_t src = trow + Ly::kPVCol + wg * DH;
      float v[2][32];
      tmem_ld32(src, v[0]);
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
        tmem_wait_ld();
        if (c + 1 < DH / 32) {
          tmem_ld32(src + 32 * (c + 1), v[(c + 1) & 1]);
        } else {
          tc_fence_before();
          mbar_arrive(pv_free);  // every column of the accumulator is read
        }
        const float(&x)[32] = v[c & 1];
        if constexpr (kDbg) {
          // this group's Wq x Vq for this warpgroup's dims (exact integers in fp32)
          if (valid) {
            int32_t* prow = p.dbg_pv + (((size_t)j * Hq + hq) * ngt + (g_begin + h)) * D + wg * DH + 32 * c;
#pragma unroll
            for (int i = 0; i < 32; ++i) prow[i] = __float2int_rn(x[i]);
          }
        }
        const uint64_t e2 = f2(e, e);
        if (rescale) {
          const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            f2_split(fma2(f2(x[2 * i], x[2 * i + 1]), e2, mul2(f2(o[32 * c + 2 * i], o[32 * c + 2 * i + 1]), a2)),
                     o[32 * c + 2 * i], o[32 * c + 2 * i + 1]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            f2_split(fma2(f2(x[2 * i], x[2 * i + 1]), e2, f2(o[32 * c + 2 * i], o[32 * c + 2 * i + 1])),
                     o[32 * c + 2 * i], o[32 * c + 2 * i + 1]);
        }
      }
    };

    for (int g = 0; g < ng; ++g) {
      if ((g & 1) == wg) softmax(g);
      if (g >= 1) update(g - 1);
    }
    if (ng >= 1) update(ng - 1);

    // ---- finish: O = o / l (both warpgroups hold the same l), or this part's
    // unnormalized (o, m, l) for the merge ----
    if (valid && nparts > 1) {
      float* ps = p.part + ((size_t)(blockIdx.x - p.full_items) * kRows + row) * (D + 4);
#pragma unroll
      for (int i = 0; i < DH / 4; ++i)
        reinterpret_cast<float4*>(ps + wg * DH)[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
      if (wg == 0) {
        ps[D] = m;
        ps[D + 1] = l;
      }
    } else if (valid) {
      const float inv = 1.0f / l;
      const size_t orow = ((size_t)j * Hq + hq) * D + wg * DH;
#pragma unroll
      for (int i = 0; i < DH / 4; ++i)
        store_out4(p.out, p.out_bf16, orow + 4 * i,
                   make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, Ly::kTmemCols);
  }
}

// The split row blocks' parts, merged by log-sum-exp: one CTA of D/4 threads
// per (split block, row), each thread one float4 column.  A part's (o, m, l) is
// unnormalized, m in log2 units; a part that saw no key of the row has
// m = -inf, l = 0 and o = 0.
template <int D>
__global__ void __launch_bounds__(D / 4) prefix_merge_kernel(PrefixParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const int tb = blockIdx.x / kRows, row = blockIdx.x % kRows;
  const int blk = p.full_items + tb;
  const int kvh = blk % p.Hkv;
  const int r = (p.nrb - 1 - blk / p.Hkv) * kRows + row;
  if (r >= p.C * p.G) return;
  const int j = r / p.G, hq = kvh * p.G + r % p.G;
  const int k = p.split_k, col = threadIdx.x;
  const float* base = p.part + ((size_t)tb * k * kRows + row) * (D + 4);
  constexpr int kMaxParts = 8;
  float mp[kMaxParts], lp[kMaxParts];
  float4 op[kMaxParts];
  float M = -INFINITY;
#pragma unroll
  for (int q = 0; q < kMaxParts; ++q) {
    if (q < k) {
      const float* ps = base + (size_t)q * kRows * (D + 4);
      op[q] = reinterpret_cast<const float4*>(ps)[col];
      mp[q] = ps[D];
      lp[q] = ps[D + 1];
      M = fmaxf(M, mp[q]);
    }
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
#pragma unroll
  for (int q = 0; q < kMaxParts; ++q) {
    if (q < k && mp[q] != -INFINITY) {
      const float w = ex2(__fsub_rn(mp[q], M));
      acc.x = __fmaf_rn(op[q].x, w, acc.x);
      acc.y = __fmaf_rn(op[q].y, w, acc.y);
      acc.z = __fmaf_rn(op[q].z, w, acc.z);
      acc.w = __fmaf_rn(op[q].w, w, acc.w);
      den = __fmaf_rn(lp[q], w, den);
    }
  }
  const float inv = 1.0f / den;
  store_out4(p.out, p.out_bf16, ((size_t)j * p.Hq + hq) * D + 4 * col,
             make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
}

constexpr int kMaxSplit = 6;

// The number of SMs of the current device (the work split depends on it).
static int device_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  return n;
}

// The last wave's split: with RB row blocks (one CTA each, one CTA per SM)
// and N SMs, the tail RB mod N blocks would run with the rest of the SMs idle.
// Each tail block is split into k parts over its key groups, k <= kMaxSplit
// and tail * k <= 2 N (the workspace bound), choosing the k that minimizes the
// tail's waves of parts per part: ceil(tail k / N) / k.  k = 1: no split.
static void choose_split(int RB, int nsm, int& full_items, int& k) {
  const int tail = RB > nsm ? RB % nsm : 0;
  k = 1;
  if (tail > 0) {
    double best = 1.0;
    for (int kk = 2; kk <= kMaxSplit && tail * kk <= 2 * nsm; ++kk) {
      const double cost = (double)((tail * kk + nsm - 1) / nsm) / kk;
      if (cost < best - 1e-9) {
        best = cost;
        k = kk;
      }
    }
  }
  full_items = k > 1 ? RB - tail : RB;
}

template <int D, bool kBF, bool kDbg = false>
cudaError_t launch_prefix_d(const PrefixParams& p0, cudaStream_t stream) {
  PrefixParams p = p0;
  const int ngt = (p.H + p.C + kGroup - 1) / kGroup;
  cudaError_t e = kBF ? launch_pdl(prefix_tiles_bf16_kernel<D>, dim3(ngt, p.Hkv), dim3(256), 0, stream, p)
                      : launch_pdl(prefix_tiles_kernel<D>, dim3(ngt, p.Hkv), dim3(256), 0, stream, p);
  if (e != cudaSuccess) return e;
  // the shared-memory opt-in, once per device (graph captures then make no attribute call)
  int dev = 0;
  cudaGetDevice(&dev);
  static bool opted[64] = {false};
  if (dev < 0 || dev >= 64 || !opted[dev]) {
    e = cudaFuncSetAttribute(prefix_attn_kernel<D, kBF, kDbg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay<D>::kTotal);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) opted[dev] = true;
  }
  const int R = p.C * p.G;
  p.nrb = (R + kRows - 1) / kRows;
  const int RB = p.nrb * p.Hkv;
  choose_split(RB, device_sms(), p.full_items, p.split_k);
  const int tail = RB - p.full_items;
  p.part = reinterpret_cast<float*>(p.tiles + (size_t)ngt * p.Hkv * Tile<D>::kBytes);
  e = launch_pdl(prefix_attn_kernel<D, kBF, kDbg>, dim3(p.full_items + tail * p.split_k), dim3(kThreads), Lay<D>::kTotal,
                 stream, p);
  if (e != cudaSuccess || tail == 0) return e;
  return launch_pdl(prefix_merge_kernel<D>, dim3(tail * kRows), dim3(D / 4), 0, stream, p);
}

}  // namespace

size_t prefix_workspace_bytes(int H, int C, int Hkv, int D) {
  const size_t ngt = ((size_t)H + C + kGroup - 1) / kGroup;
  const size_t tiles = ngt * Hkv * (D == 256 ? Tile<256>::kBytes : Tile<128>::kBytes);
  // the split parts' (o, m, l): at most 2 x #SM parts of 128 rows
  return tiles + (size_t)2 * device_sms() * kRows * (D + 4) * sizeof(float);
}

cudaError_t launch_int8_prefix(const PrefixParams& p, cudaStream_t stream) {
  return p.D == 256 ? launch_prefix_d<256, false>(p, stream) : launch_prefix_d<128, false>(p, stream);
}

cudaError_t launch_bf16_prefix(const PrefixParams& p, cudaStream_t stream) {
  return p.D == 256 ? launch_prefix_d<256, true>(p, stream) : launch_prefix_d<128, true>(p, stream);
}

cudaError_t launch_debug_prefix(const PrefixParams& p, cudaStream_t stream) {
  // the records cover only the keys each row sees: clear them first
  const size_t ng = ((size_t)p.H + p.C + kGroup - 1) / kGroup;
  const size_t rows = (size_t)p.C * p.Hq;
  cudaError_t e = cudaMemsetAsync(p.dbg_s, 0, rows * (p.H + p.C) * sizeof(int32_t), stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(p.dbg_wq, 0, rows * ng * kGroup, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(p.dbg_pv, 0, rows * ng * p.D * sizeof(int32_t), stream);
  if (e != cudaSuccess) return e;
  return p.D == 256 ? launch_prefix_d<256, false, true>(p, stream) : launch_prefix_d<128, false, true>(p, stream);
}

}  // namespace i8kv
