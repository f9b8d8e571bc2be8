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
//   S  = Qq x Kq^T        tcgen05, M = 128, N = 64 (two groups at once), K = D,
//                         the query codes (A) held in tensor memory, into TMEM
//   scores, causal mask, p~ = exp(s - m_g) against the group's own row
//   maximum m_g, W = p~ sV, sW = max W / 127, Wq = round(W / sW)
//                         CUDA cores, one thread per row
//   PV = Wq x Vq          tcgen05, M = 128, N = D / 2 per half, K = 32, into TMEM
//   o  = alpha o + exp(m_g - m) sW PV,  l = alpha l + exp(m_g - m) l_g
//                         CUDA cores, o in registers (half of D per thread)
// where m is the row's reference maximum.  The codes round(W / sW) do not
// change when W is scaled, so quantizing each group against m_g and bringing it
// to the reference maximum in the output update is the pages' online softmax,
// reordered; it lets the softmax of a group start before the previous group's
// maximum is known.  The reference maximum moves only when a group's maximum
// passes it by more than 2^8 (alpha = 1 otherwise), so o is rarely rescaled.
// Scores are kept in log2 units (the scale folds in log2 e) so every
// exponential is one ex2.
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
// by the group's sK and sV.  The attention kernel moves a tile with D/64 + 1
// bulk copies: K into a ring of its own, atom-major, so the K rows of two
// adjacent stages form one 64-key operand, and V with the scales into a second
// ring.  Each row block starts its walk over the key groups at its own hashed
// offset and wraps around, so the CTAs that run together on one KV head read
// different tiles.
//
// Warps of the attention kernel (512 threads, one CTA per SM):
//   warp 0      the tile copies (one lane per copy)
//   warp 1      lane 0 issues the QK MMAs of each pair of groups into one of two
//               64-column S slots; the warp owns the TMEM allocation
//   warp 2      lane 0 issues the PV MMAs, each group as two halves of D / 2
//               columns, one per update warpgroup
//   warps 4-11  two update warpgroups, one half of D each: o, l per row
//   warps 12-15 the softmax warpgroup: loads the query rows into TMEM, then the
//               softmax of every group (thread = row), handing the f16 codes
//               (a swizzled Wq tile) and (m_g, sW, l_g) to the PV issuer and
//               the update warpgroups
// so the softmax of group g + 1 runs while the update warpgroups apply group g.
// setmaxnreg splits the registers 40 / 184 / 184 / 104 between the control
// warps, the update warpgroups and the softmax warpgroup.
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
constexpr int kThreads = 512;
constexpr int kLoadWarp = 0;
constexpr int kMmaWarp = 1;      // issues the QK MMAs
constexpr int kPvWarp = 2;       // issues the PV MMAs
constexpr int kUpdWarp0 = 4;     // warps 4..11: output update, warpgroup 1 = dims [0, D/2), 2 = [D/2, D)
constexpr int kSmxWarp0 = 12;    // warps 12..15: the softmax of every group
constexpr int kWGThreads = 128;
// Register split (setmaxnreg) of the launch's 512 x 128 registers: copy/MMA
// warpgroup 40, update warpgroups 184 each (o is D/2 fp32 per thread), softmax
// warpgroup 104; 40 + 2 x 184 + 104 = 4 x 128.
constexpr int kRegsCtl = 40, kRegsUpd = 184, kRegsSmx = 104;
static_assert(kRegsCtl + 2 * kRegsUpd + kRegsSmx == 4 * (65536 / kThreads), "register split");
// TMEM columns per load in the output update.
constexpr int kUpdChunk = 32;
template <int N>
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, float (&v)[N]) {
  if constexpr (N == 8)
    tmem_ld8(taddr, v);
  else if constexpr (N == 16)
    tmem_ld16(taddr, v);
  else
    tmem_ld32(taddr, v);
}
// The output's reference maximum moves only when a group's maximum exceeds it
// by more than this (log2 units), so o is rarely rescaled.
constexpr float kLazyLog2 = 8.0f;

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
  // Operand tiles in flight (an even number: QK takes the keys of two
  // consecutive groups at once).  K goes to a ring of its own, atom-major --
  // [D/64 atoms][kStages][32 keys][128 B] -- so the K rows of two adjacent
  // stages are one 64-row operand; V and the scales go to a ring of stages.
  static constexpr int kStages = D == 256 ? 6 : 8;
  static constexpr int kKAtom = kGroup * 128;         // one stage's 32 rows of one 64-dim atom
  static constexpr int kVBytes = Tile<D>::kBytes - Tile<D>::oV;  // V, then sK, sV
  static constexpr int kVSlot = (kVBytes + 1023) / 1024 * 1024;
  static constexpr int kP16 = kRows * kGroup * 2;     // f16 Wq, [128][64 B]
  static constexpr int oK = 0;                        // the K ring
  static constexpr int oVr = oK + (D / 64) * kStages * kKAtom;  // the V ring
  static constexpr int oP = oVr + kStages * kVSlot;   // two slots
  static constexpr int oSt = oP + 2 * kP16;           // four slots of m_g[128], sW[128], l_g[128]
  static constexpr int oBar = oSt + 4 * 3 * kRows * 4;
  // tile_full[4], tile_free[4], qk_done[2], s_free[2], p_full[2], wq_free[2], pv_done[2], pv_free[2], st_full[4]
  static constexpr int kBars = kStages + kStages + 2 + 2 + 2 + 2 + 2 + 2 + 4;
  static constexpr int oCtl = oBar + kBars * 8;       // TMEM base, abort flag
  static constexpr int kTotal = oCtl + 16;
  // TMEM: S in columns [0, 128) (two slots of 64: a pair of groups each), the
  // f16 query (the QK MMAs' A operand, D / 2 columns) in [kQCol, kPVCol), PV in
  // [kPVCol, kPVCol + D)
  static constexpr uint32_t kPVCol = 256;
  static constexpr uint32_t kQCol = kPVCol - D / 2;
  static constexpr uint32_t kTmemCols = 512;
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
  // K page [D/16][16 tokens][16 B] -> [key][D] (SW128 atoms): chunk i = (page, dim chunk, token);
  // V page [D][16 tokens] -> [D][32 keys] (SW64): chunk i = (page, dim).  Every
  // thread loads all of its chunks before it stores any, so the loads are in
  // flight together.
  constexpr int KC = kPagesPG * (D / 16) * kBS, VC = kPagesPG * D;
  static_assert(KC % 256 == 0 && VC % 256 == 0, "whole chunks per thread");
  uint4 kv[KC / 256], vv[VC / 256];
#pragma unroll
  for (int j = 0; j < KC / 256; ++j) {
    const int i = tid + 256 * j;
    const int pg = i / ((D / 16) * kBS), rem = i % ((D / 16) * kBS);
    kv[j] = blk[pg] >= 0
                ? __ldg(reinterpret_cast<const uint4*>(p.k_cache + ((size_t)blk[pg] * Hkv + kvh) * (D * kBS)) + rem)
                : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int j = 0; j < VC / 256; ++j) {
    const int i = tid + 256 * j;
    const int pg = i / D, d = i % D;
    vv[j] = blk[pg] >= 0
                ? __ldg(reinterpret_cast<const uint4*>(p.v_cache + ((size_t)blk[pg] * Hkv + kvh) * (D * kBS)) + d)
                : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int j = 0; j < KC / 256; ++j) {
    const int i = tid + 256 * j;
    const int pg = i / ((D / 16) * kBS), rem = i % ((D / 16) * kBS);
    const int dc = rem / kBS, key = pg * kBS + rem % kBS;
    uint4 h0, h1;
    s8x16_to_f16(kv[j], h0, h1);
    uint8_t* atom = tile + T::oK + (size_t)(dc / 4) * (kGroup * 128);
    *reinterpret_cast<uint4*>(atom + swz_chunk<128>(key, 2 * (dc % 4))) = h0;
    *reinterpret_cast<uint4*>(atom + swz_chunk<128>(key, 2 * (dc % 4) + 1)) = h1;
  }
#pragma unroll
  for (int j = 0; j < VC / 256; ++j) {
    const int i = tid + 256 * j;
    const int pg = i / D, d = i % D;
    uint4 h0, h1;
    s8x16_to_f16(vv[j], h0, h1);
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

// ---- bf16 operand tiles from the BF16 paged cache (the BF16-KV comparison of
// the prefix chunk): one CTA per (group, KV head).  Every key, history and
// chunk alike, comes from the bf16 cache (K [NB, Hkv, D/8, 16, 8], V [NB, Hkv,
// D, 16]) through block_table; keys past the sequence are zero (their cache
// slots may hold anything, and a NaN there would reach the P x V sums).
template <int D>
__global__ void __launch_bounds__(256) prefix_tiles_bf16kv_kernel(PrefixParams p) {
  using T = Tile<D>;
  griddep_wait();
  griddep_launch_dependents();
  const int g = blockIdx.x, kvh = blockIdx.y, tid = threadIdx.x;
  const int Hkv = p.Hkv, n = p.H + p.C;
  const int key0 = g * kGroup;
  uint8_t* tile = p.tiles + ((size_t)kvh * gridDim.x + g) * T::kBytes;
  int blk[kPagesPG];
#pragma unroll
  for (int i = 0; i < kPagesPG; ++i) {
    const int lb = g * kPagesPG + i;
    blk[i] = -1;
    if (lb * kBS < n) {
      const int b = p.block_table[lb];
      if (b < 0 || b >= p.num_blocks) {
        if (tid == 0) record_error(2);
      } else {
        blk[i] = b;
      }
    }
  }
  const uint16_t* kc = p.kb_cache;
  const uint16_t* vc = p.vb_cache;
  // K: (page, 8-dim chunk, token) -> one 16-byte chunk of row `key` (SW128 atoms of 64 dims)
  for (int i = tid; i < kPagesPG * (D / 8) * kBS; i += 256) {
    const int pg = i / ((D / 8) * kBS), rem = i % ((D / 8) * kBS);
    const int c8 = rem / kBS, tok = rem % kBS, key = pg * kBS + tok;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (blk[pg] >= 0 && key0 + key < n)
      v = __ldg(reinterpret_cast<const uint4*>(kc + ((size_t)blk[pg] * Hkv + kvh) * (D * kBS)) + rem);
    uint8_t* atom = tile + T::oK + (size_t)(c8 / 8) * (kGroup * 128);
    *reinterpret_cast<uint4*>(atom + swz_chunk<128>(key, c8 % 8)) = v;
  }
  // V: (page, dim) -> the page's 16 tokens of that dim, chunks 2 pg and 2 pg + 1 of row d (SW64)
  for (int i = tid; i < kPagesPG * D; i += 256) {
    const int pg = i / D, d = i % D;
    uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
    if (blk[pg] >= 0) {
      const uint4* src = reinterpret_cast<const uint4*>(vc + (((size_t)blk[pg] * Hkv + kvh) * D + d) * kBS);
      h0 = __ldg(src);
      h1 = __ldg(src + 1);
      const int valid = n - (key0 + pg * kBS);  // tokens of this page inside the sequence
      if (valid < kBS) {
        uint32_t w[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (2 * e >= valid) w[e] = 0u;
          else if (2 * e + 1 >= valid) w[e] &= 0xffffu;
        }
        h0 = make_uint4(w[0], w[1], w[2], w[3]);
        h1 = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
    *reinterpret_cast<uint4*>(tile + T::oV + swz_chunk<64>(d, 2 * pg)) = h0;
    *reinterpret_cast<uint4*>(tile + T::oV + swz_chunk<64>(d, 2 * pg + 1)) = h1;
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
  constexpr int DH = D / 2;  // output dims per update warpgroup (one PV half)
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* tile_full = reinterpret_cast<uint64_t*>(smem + Ly::oBar);  // [g % Ly::kStages]: tile g landed
  uint64_t* tile_free = tile_full + Ly::kStages;  // [g % Ly::kStages]: PV(g) done, the tile slot may be refilled
  uint64_t* qk_done = tile_free + Ly::kStages;    // [g & 1]: S(g) in TMEM
  uint64_t* s_free = qk_done + 2;             // [g & 1]: S(g) read
  uint64_t* p_full = s_free + 2;              // [g & 1]: Wq(g) in its slot
  uint64_t* wq_free = p_full + 2;             // [g & 1]: PV(g) done (both halves), the Wq slot may be rewritten
  uint64_t* pv_done = wq_free + 2;            // [half]: PV(g) of that half in TMEM
  uint64_t* pv_free = pv_done + 2;            // [half]: that half of the accumulator read
  uint64_t* st_full = pv_free + 2;            // [g & 3]: the group's row statistics
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
  // The online softmax takes the key groups in any order, so each row block
  // starts its walk at its own (hashed) offset and wraps around: the CTAs that
  // run at the same time on one KV head then read different operand tiles,
  // instead of all asking L2 for the same tile at once.
  const int rot = ng > 0 ? (int)(((unsigned)(blk / p.Hkv) * 2654435761u >> 7) % (unsigned)ng) : 0;
  auto gid = [&](int g) { return g_begin + (g + rot < ng ? g + rot : g + rot - ng); };

  if (tid == 0) {
    for (int s = 0; s < Ly::kStages; ++s) {
      mbar_init(&tile_full[s], 1);
      mbar_init(&tile_free[s], 1);
    }
    for (int s = 0; s < 4; ++s) mbar_init(&st_full[s], kWGThreads);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qk_done[s], 1);
      mbar_init(&s_free[s], 2 * kWGThreads);  // both groups of a pair
      mbar_init(&p_full[s], kWGThreads);
      mbar_init(&wq_free[s], 1);
      mbar_init(&pv_done[s], 1);
      mbar_init(&pv_free[s], kWGThreads);
    }
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

  // ---- the f16 query rows -> TMEM (the softmax warpgroup: thread = row), the
  // QK MMAs' A operand; row r of the block in lane r, two elements per column ----
  if (warp >= kSmxWarp0) {
    const int qrow = (warp & 3) * 32 + lane;
    const int r = r0 + qrow;
    const uint32_t qt = tmem + ((uint32_t)((warp & 3) * 32) << 16) + Ly::kQCol;
#pragma unroll 1
    for (int c = 0; c < D / 64; ++c) {  // 64 elements = 32 columns at a time
      uint32_t w[32];
      if constexpr (kBF) {
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = make_uint4(0, 0, 0, 0);
        if (r < R) {
          const int j = r / G, hq = kvh * G + r % G;
          const uint4* src = reinterpret_cast<const uint4*>(p.qb + ((size_t)j * Hq + hq) * D + 64 * c);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = __ldg(src + i);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          w[4 * i] = v[i].x;
          w[4 * i + 1] = v[i].y;
          w[4 * i + 2] = v[i].z;
          w[4 * i + 3] = v[i].w;
        }
      } else {
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = make_uint4(0, 0, 0, 0);
        if (r < R) {
          const int j = r / G, hq = kvh * G + r % G;
          const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)j * Hq + hq) * D + 64 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i) v[i] = __ldg(src + i);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 h0, h1;
          s8x16_to_f16(v[i], h0, h1);
          w[8 * i] = h0.x;
          w[8 * i + 1] = h0.y;
          w[8 * i + 2] = h0.z;
          w[8 * i + 3] = h0.w;
          w[8 * i + 4] = h1.x;
          w[8 * i + 5] = h1.y;
          w[8 * i + 6] = h1.z;
          w[8 * i + 7] = h1.w;
        }
      }
      tmem_st32(qt + 32 * c, w);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // this thread's query row (softmax and update warpgroups: one TMEM lane each)
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const int r = r0 + row;
  const bool valid = r < R;
  const int j = valid ? r / G : 0, hq = kvh * G + (valid ? r % G : 0);
  const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
  float* stats = reinterpret_cast<float*>(smem + Ly::oSt);  // [slot][m_g | sW | l_g][row]

  if (warp < kUpdWarp0) {
    regs_dec<kRegsCtl>();  // the copy and MMA warps hand registers to the others
    if (warp == kLoadWarp) {
      // ================= tile copies (warp 0) =================
      // A tile is D/64 K atoms of 4 KB, each into its row of the K ring, and
      // the V tile with the scales behind it, into the V ring: one bulk copy
      // per lane.
      constexpr int kCopies = D / 64 + 1;
      const uint8_t* src = p.tiles + (size_t)kvh * ngt * T::kBytes;
      int g = 0;
      for (; g < ng; ++g) {
        const int st = g % Ly::kStages;
        if (g >= Ly::kStages) pwait(&tile_free[st], ((g - Ly::kStages) / Ly::kStages) & 1, abort_flag);
        if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        if (lane == 0) mbar_expect_tx(&tile_full[st], T::kBytes);
        __syncwarp();
        const uint8_t* tsrc = src + (size_t)gid(g) * T::kBytes;
        if (lane < D / 64)
          bulk_g2s(smem + Ly::oK + ((size_t)lane * Ly::kStages + st) * Ly::kKAtom, tsrc + T::oK + lane * Ly::kKAtom,
                   Ly::kKAtom, &tile_full[st]);
        else if (lane == D / 64)
          bulk_g2s(smem + Ly::oVr + (size_t)st * Ly::kVSlot, tsrc + T::oV, Ly::kVBytes, &tile_full[st]);
        static_assert(kCopies <= 32, "one copy per lane");
        __syncwarp();
        if (lane == 0) mbar_arrive(&tile_full[st]);
      }
      // copies issued but never waited for (after an abort) land before the CTA exits
      if (lane == 0)
        for (int k = max(0, g - Ly::kStages); k < g; ++k) mbar_wait(&tile_full[k % Ly::kStages], (k / Ly::kStages) & 1);
    } else if ((warp == kMmaWarp || warp == kPvWarp) && lane == 0) {
      // ================= MMA issue (warp 1: QK; warp 2: PV; lane 0 each) =================
      // Two issuing threads, so that issuing one kind never holds up the other
      // (a tcgen05.mma takes a while to be accepted).  The checks never suspend
      // (test_wait); an idle pass spins (a sleep delayed the next issue by most
      // of a microsecond), with the abort flag and the time limit checked every
      // 64 idle passes.  A group's PV runs as two halves of D/2 columns, one
      // per update warpgroup, so each half waits only for its own warpgroup's
      // read of the previous group; the high half of a group follows its low half.
      constexpr uint32_t idesc_qk = kBF ? umma_idesc_bf16(kRows, 2 * kGroup) : umma_idesc_f16(kRows, 2 * kGroup);
      constexpr uint32_t idesc_pv = kBF ? umma_idesc_bf16(kRows, DH) : umma_idesc_f16(kRows, DH);
      const uint32_t kring = smem_u32(smem + Ly::oK), vring = smem_u32(smem + Ly::oVr);
      const bool qk = warp == kMmaWarp;
      int nq = 0, np[2] = {0, 0};  // next QK pair's first group; next PV of each half
      uint64_t* last_bar = nullptr;  // this thread's latest commit (it completes after its earlier MMAs)
      uint32_t last_par = 0;
      uint64_t t_idle = 0;
      uint32_t idle = 0;
      while (qk ? nq < ng : np[1] < ng) {
        bool did = false;
        if (qk) {
          // QK of the pair of groups (nq, nq + 1), nq even: their K rows are
          // adjacent in the K ring (N = 64); a last group without a partner
          // still runs as a pair (its partner's half of S is never read)
          if (mbar_test(&tile_full[nq % Ly::kStages], (nq / Ly::kStages) & 1) &&
              (nq + 1 >= ng || mbar_test(&tile_full[(nq + 1) % Ly::kStages], ((nq + 1) / Ly::kStages) & 1)) &&
              (nq < 4 || mbar_test(&s_free[(nq >> 1) & 1], ((nq - 4) >> 2) & 1))) {
            const uint32_t k16 = kring + (nq % Ly::kStages) * Ly::kKAtom;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t b = k16 + (kk / 4) * (Ly::kStages * Ly::kKAtom) + (kk % 4) * 32;
              umma_f16_ta(tmem + 64 * ((nq >> 1) & 1), tmem + Ly::kQCol + 8 * kk, umma_desc(b, 128), idesc_qk,
                          kk > 0);
            }
            umma_commit(&qk_done[(nq >> 1) & 1]);
            last_bar = &qk_done[(nq >> 1) & 1];
            last_par = (nq >> 2) & 1;
            nq += 2;
            did = true;
          }
        } else {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int g = np[hf];
            if (g < ng && (hf == 0 || g < np[0]) && mbar_test(&p_full[g & 1], (g >> 1) & 1) &&
                (g < 1 || mbar_test(&pv_free[hf], (g - 1) & 1))) {
              const uint32_t p16 = smem_u32(smem + Ly::oP + (size_t)(g & 1) * Ly::kP16);
              // V tile rows (head dims) [hf DH, (hf + 1) DH): a whole number of SW64 atoms further on
              const uint32_t v16 = vring + (g % Ly::kStages) * Ly::kVSlot + hf * DH * 64;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < kGroup / 16; ++kk)
                umma_f16(tmem + Ly::kPVCol + hf * DH, umma_desc(p16 + kk * 32, 64), umma_desc(v16 + kk * 32, 64),
                         idesc_pv, kk > 0);
              umma_commit(&pv_done[hf]);
              last_bar = &pv_done[hf];
              last_par = g & 1;
              if (hf == 1) {
                umma_commit(&wq_free[g & 1]);
                umma_commit(&tile_free[g % Ly::kStages]);
                last_bar = &wq_free[g & 1];
                last_par = (g >> 1) & 1;
              }
              ++np[hf];
              did = true;
            }
          }
        }
        if (did) {
          t_idle = 0;
          idle = 0;
        } else if ((++idle & 63) == 0) {
          if (*abort_flag) break;
          const uint64_t now = global_timer_ns();
          if (t_idle == 0) {
            t_idle = now;
          } else if (now - t_idle > kWaitLimitNs) {
            record_error(1);
            *abort_flag = 1;
            break;
          }
        }
      }
      // every MMA this thread issued has completed before TMEM is released
      if (last_bar) mbar_wait(last_bar, last_par);
    }
    __syncwarp();
  } else if (warp < kSmxWarp0) {
    // ================= output update (warpgroups 1, 2: one PV half each) =================
    regs_inc<kRegsUpd>();
    const int hf = (warp - kUpdWarp0) >> 2;
    float o[DH];
#pragma unroll
    for (int i = 0; i < DH; ++i) o[i] = 0.f;
    float m = -INFINITY, l = 0.f;  // m: the reference maximum o and l are scaled to (log2 units)
    const uint32_t src = trow + Ly::kPVCol + hf * DH;
    for (int g = 0; g < ng; ++g) {
      // o = alpha o + 2^(m_g - m) sW (Wq x Vq), l = alpha l + 2^(m_g - m) l_g.  The
      // reference maximum moves only when a group's maximum exceeds it by more than
      // kLazyLog2 (then alpha = 2^(m - m_g)); otherwise alpha = 1 and the group's
      // factor is at most 2^kLazyLog2, so o is rescaled only a few times per row.
      pwait(&pv_done[hf], g & 1, abort_flag);
      pwait(&st_full[g & 3], (g >> 2) & 1, abort_flag);
      const float* st = stats + (g & 3) * 3 * kRows;
      const float mg = st[row], sw = st[kRows + row], lg = st[2 * kRows + row];
      float alpha = 1.f, e = 0.f;
      if (mg != -INFINITY) {
        if (mg > m + kLazyLog2) {  // also the first group (m = -inf)
          alpha = m == -INFINITY ? 0.f : ex2(__fsub_rn(m, mg));
          l = __fmul_rn(l, alpha);
          m = mg;
        }
        const float f = ex2(__fsub_rn(mg, m));
        e = __fmul_rn(f, sw);
        l = __fmaf_rn(lg, f, l);
      }
      tc_fence_after();
      const bool rescale = __any_sync(0xffffffffu, alpha != 1.f);
      // kCh-column chunks, two in flight: chunk c + 1 is loading while chunk c
      // joins the output (tcgen05.wait::ld waits for every load issued so far)
      // kCh-column chunks, one load in flight: the round trips, not the few
      // fused multiply-adds between them, set the pace, so the widest load the
      // registers allow (o takes D/2 of them) comes first
      constexpr int kCh = kUpdChunk;
#pragma unroll
      for (int c = 0; c < DH / kCh; ++c) {
        float x[kCh];
        tmem_ld_chunk(src + kCh * c, x);
        tmem_wait_ld();
        if (c + 1 == DH / kCh) {
          tc_fence_before();
          mbar_arrive(&pv_free[hf]);  // every column of this half is read
        }
        if constexpr (kDbg) {
          // this group's Wq x Vq for this half's dims (exact integers in fp32)
          if (valid) {
            int32_t* prow = p.dbg_pv + (((size_t)j * Hq + hq) * ngt + gid(g)) * D + hf * DH + kCh * c;
#pragma unroll
            for (int i = 0; i < kCh; ++i) prow[i] = __float2int_rn(x[i]);
          }
        }
        const uint64_t e2 = f2(e, e);
        if (rescale) {
          const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
          for (int i = 0; i < kCh / 2; ++i)
            f2_split(fma2(f2(x[2 * i], x[2 * i + 1]), e2, mul2(f2(o[kCh * c + 2 * i], o[kCh * c + 2 * i + 1]), a2)),
                     o[kCh * c + 2 * i], o[kCh * c + 2 * i + 1]);
        } else {
#pragma unroll
          for (int i = 0; i < kCh / 2; ++i)
            f2_split(fma2(f2(x[2 * i], x[2 * i + 1]), e2, f2(o[kCh * c + 2 * i], o[kCh * c + 2 * i + 1])),
                     o[kCh * c + 2 * i], o[kCh * c + 2 * i + 1]);
        }
      }
    }
    // ---- finish: O = o / l (both warpgroups hold the same l), or this part's
    // unnormalized (o, m, l) for the merge ----
    if (valid && nparts > 1) {
      float* ps = p.part + ((size_t)(blockIdx.x - p.full_items) * kRows + row) * (D + 4);
#pragma unroll
      for (int i = 0; i < DH / 4; ++i)
        reinterpret_cast<float4*>(ps + hf * DH)[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
      if (hf == 0) {
        ps[D] = m;
        ps[D + 1] = l;
      }
    } else if (valid) {
      const float inv = 1.0f / l;
      const size_t orow = ((size_t)j * Hq + hq) * D + hf * DH;
#pragma unroll
      for (int i = 0; i < DH / 4; ++i)
        store_out4(p.out, p.out_bf16, orow + 4 * i,
                   make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv));
    }
  } else {
    // ================= softmax of every group (warpgroup 3) =================
    regs_dec<kRegsSmx>();
    const int lim = valid ? H + j : -1;  // last visible key
    // score in log2 units: acc x sK x (sQ x scale x log2(e))
    const float c2 = !valid ? 0.f
                     : kBF  ? __fmul_rn(p.sm_scale, kLog2e)
                            : __fmul_rn(__fmul_rn(p.q_scale[(size_t)j * Hq + hq], p.sm_scale), kLog2e);
    const uint64_t c2p = f2(c2, c2);
    for (int g = 0; g < ng; ++g) {
      const int sl = g & 1;
      pwait(&qk_done[(g >> 1) & 1], (g >> 2) & 1, abort_flag);
      tc_fence_after();
      float s[32];
      tmem_ld32(trow + 64 * ((g >> 1) & 1) + 32 * sl, s);
      const int key0 = gid(g) * kGroup;
      const bool full = __all_sync(0xffffffffu, key0 + kGroup - 1 <= lim);  // no key of the warp is masked
      float mg = -INFINITY, lg = 0.f, sw = 0.f;
      uint32_t pk[16];
      // x = acc x sK (INT8) or acc (BF16); m_g = c2 max x (c2 >= 0, so rounding
      // keeps the order); p~ = 2^(x c2 - m_g), one fused multiply-add per key;
      // a masked key has x = -inf and p~ = 0.
      const float4* sk4 = nullptr;
      if constexpr (!kBF) {
        pwait(&tile_full[g % Ly::kStages], (g / Ly::kStages) & 1, abort_flag);  // the group's scales (already landed)
        sk4 = reinterpret_cast<const float4*>(smem + Ly::oVr + (size_t)(g % Ly::kStages) * Ly::kVSlot +
                                              (T::oSk - T::oV));
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&s_free[(g >> 1) & 1]);  // S is in registers; the QK of the pair after next may overwrite it
      if constexpr (kDbg) {
        // the raw accumulators of the visible keys (exact integers in fp32)
        if (valid) {
          int32_t* srow = p.dbg_s + ((size_t)j * Hq + hq) * (H + C);
#pragma unroll
          for (int t = 0; t < 32; ++t)
            if (key0 + t <= lim) srow[key0 + t] = __float2int_rn(s[t]);
        }
      }
      if constexpr (!kBF) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 k4 = sk4[i];
          f2_split(mul2(f2(s[4 * i], s[4 * i + 1]), f2(k4.x, k4.y)), s[4 * i], s[4 * i + 1]);
          f2_split(mul2(f2(s[4 * i + 2], s[4 * i + 3]), f2(k4.z, k4.w)), s[4 * i + 2], s[4 * i + 3]);
        }
      }
      if (!full) {
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (key0 + t > lim) s[t] = -INFINITY;
      }
      const float mx = tree_max(s);
      float A = 0.f;
      if (mx != -INFINITY) {
        mg = __fmul_rn(mx, c2);
        const uint64_t nm = f2(-mg, -mg);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float lo, hi;
          f2_split(fma2(f2(s[2 * i], s[2 * i + 1]), c2p, nm), lo, hi);
          s[2 * i] = ex2(lo);
          s[2 * i + 1] = ex2(hi);
        }
        if (!full) {  // a masked key's -inf times c2 = 0 (a zero query) would be NaN
#pragma unroll
          for (int t = 0; t < 32; ++t)
            if (key0 + t > lim) s[t] = 0.f;
        }
        lg = tree_sum(s);
        if constexpr (!kBF) {
          const float4* sv4 = sk4 + kGroup / 4;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 v4 = sv4[i];
            f2_split(mul2(f2(s[4 * i], s[4 * i + 1]), f2(v4.x, v4.y)), s[4 * i], s[4 * i + 1]);
            f2_split(mul2(f2(s[4 * i + 2], s[4 * i + 3]), f2(v4.z, v4.w)), s[4 * i + 2], s[4 * i + 3]);
          }
          A = tree_max(s);
        }
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t) s[t] = 0.f;
      }
      if constexpr (kBF) {
        sw = 1.f;
        // p~ as bf16, two per register (low half = the even key)
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = bf16x2_bits(s[2 * i], s[2 * i + 1]);
      } else {
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
            uint32_t h = __byte_perm(qb[2 * i], qb[2 * i + 1], 0x5410);
            asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(h) : "r"(0x64006400u));
            pk[i] = h;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = 0u;
        }
        if constexpr (kDbg) {
          if (valid) {
            uint8_t* wrow = p.dbg_wq + ((size_t)j * Hq + hq) * (size_t)(ngt * kGroup);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 cc = __half22float2(*reinterpret_cast<const __half2*>(&pk[i]));
              if (key0 + 2 * i <= lim) wrow[key0 + 2 * i] = (uint8_t)__float2int_rn(cc.x);
              if (key0 + 2 * i + 1 <= lim) wrow[key0 + 2 * i + 1] = (uint8_t)__float2int_rn(cc.y);
            }
          }
        }
      }
      // Wq (f16) or p~ (bf16) -> the PV A tile, row `row`; then the row statistics
      if (g >= 2) pwait(&wq_free[sl], ((g - 2) >> 1) & 1, abort_flag);  // PV(g-2) has read the slot
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
  cudaError_t e = !kBF          ? launch_pdl(prefix_tiles_kernel<D>, dim3(ngt, p.Hkv), dim3(256), 0, stream, p)
                  : p.kb_cache ? launch_pdl(prefix_tiles_bf16kv_kernel<D>, dim3(ngt, p.Hkv), dim3(256), 0, stream, p)
                               : launch_pdl(prefix_tiles_bf16_kernel<D>, dim3(ngt, p.Hkv), dim3(256), 0, stream, p);
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
