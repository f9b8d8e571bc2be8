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
//   scores, causal mask, online softmax, W = p~ sV, sW = max W / 127,
//   Wq = round(W / sW)    CUDA cores, one thread per (row, half of the keys)
//   PV = Wq x Vq          tcgen05, M = 128, N = D, K = 32, into TMEM
//   o  = alpha o + sW PV  CUDA cores, o in registers (half of D per thread)
// The int8 codes are exact in f16, every product (<= 127^2) is exact and every
// partial sum stays below 2^22, so f16 MMAs with fp32 accumulation give the
// INT8 contractions' exact integer results.
//
// Warps.  Warp 0 lane 0 issues the bulk copies of each group's int8 pages and
// scale rows (three groups in flight); warps 0, 2 and 3 convert each group
// once into f16 operand tiles (K-major, 16-byte chunks XOR-swizzled: K as
// [key][dim] in 128-byte rows, V as [dim][key] in 64-byte rows).  Warp 1 owns
// the TMEM allocation; its lane 0 issues every MMA.  Warps 4-7 and 8-11 are two
// halves: thread (half, row) takes keys 16 half .. 16 half + 15 of each group
// for its row's softmax (the halves exchange the row's group maximum and
// absmax through shared memory) and output dims [half D/2, (half + 1) D/2).
// S is double-buffered in TMEM, so the QK of the next group runs during a
// softmax; the PV of group g runs during the softmax of g + 1, after which the
// output takes group g's product.
#include "common.cuh"
#include "kernels.h"

namespace i8kv {
I8KV_DEFINE_ERROR_ACCESSOR(read_error_prefix)

namespace {

constexpr int kBS = 16;
constexpr int kRows = 128;       // query rows per CTA: the MMA's M, one TMEM lane each
constexpr int kGroup = 32;       // keys per probability group
constexpr int kPagesPG = kGroup / kBS;
constexpr int kStages = 3;       // int8 staging buffers (groups in flight)
constexpr int kMaxHkv = 8;
constexpr int kThreads = 384;
constexpr int kMmaWarp = 1;
constexpr int kCompWarp0 = 4;    // warps 4..11
constexpr int kConvThreads = 96; // warps 0, 2, 3
constexpr int kCompThreads = 256;

template <int D>
struct Lay {
  static constexpr int kQ16 = kRows * D * 2;          // f16 Q, D/64 atoms of [128 rows][128 B]
  static constexpr int kK16 = kGroup * D * 2;         // f16 K, D/64 atoms of [32 keys][128 B]
  static constexpr int kV16 = D * kGroup * 2;         // f16 V, [D][64 B]
  static constexpr int kP16 = kRows * kGroup * 2;     // f16 Wq, [128][64 B]
  static constexpr int kPage = D * kBS;               // one int8 K or V page
  static constexpr int kSRow = kBS * kMaxHkv * 4;     // one block's scale rows (room for kMaxHkv heads)
  static constexpr int kStage = 2 * kPagesPG * kPage + 2 * kPagesPG * kSRow;
  static constexpr int oQ = 0;
  static constexpr int oK = oQ + kQ16;                // two slots
  static constexpr int oV = oK + 2 * kK16;            // two slots
  static constexpr int oP = oV + 2 * kV16;            // two slots
  static constexpr int oStage = oP + 2 * kP16;        // kStages
  static constexpr int oSc = oStage + kStages * kStage;  // two slots of [32 keys][sK, sV]
  static constexpr int oX = oSc + 2 * kGroup * 8;     // exchange: [3 values][2 halves][128 rows] floats
  static constexpr int oBar = oX + 3 * 2 * kRows * 4;
  // barriers: stage_full[3], conv_full[2], s_full[2], s_free[2], p_full[2], mma_done[2], pv_free
  static constexpr int kBars = kStages + 2 + 2 + 2 + 2 + 2 + 1;
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

// Bounded wait that gives up at once when the CTA has aborted (error 1 after
// the time limit); every thread still runs the same loop and the same named
// barriers, so no thread waits on a barrier another one skipped.
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1) int8_prefix_kernel(PrefixParams p) {
  using Ly = Lay<D>;
  constexpr int DH = D / 2;  // output dims per half
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::oBar);
  uint64_t* stage_full = bars;
  uint64_t* conv_full = stage_full + kStages;
  uint64_t* s_full = conv_full + 2;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* mma_done = p_full + 2;  // PV of group g done: its slots and the PV accumulator are readable/free
  uint64_t* pv_free = mma_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::oCtl);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::oCtl + 4);
  float* xch = reinterpret_cast<float*>(smem + Ly::oX);  // [value][half][row]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.y;
  const int G = p.G, Hkv = p.Hkv, Hq = p.Hq, H = p.H, C = p.C;
  const int R = C * G;
  // Row blocks in reverse: later chunk tokens see more keys, and CTAs start in
  // index order, so the heaviest blocks run first and the last wave holds the
  // lightest ones.
  const int r0 = (gridDim.x - 1 - blockIdx.x) * kRows;
  const int j_hi = min(C - 1, (r0 + kRows - 1) / G);
  const int n_keys = H + j_hi + 1;
  const int ng = (n_keys + kGroup - 1) / kGroup;
  const int max_blk = (H + C + kBS - 1) / kBS;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&stage_full[s], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&conv_full[s], kConvThreads);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], kCompThreads);
      mbar_init(&p_full[s], kCompThreads);
      mbar_init(&mma_done[s], 1);
    }
    mbar_init(pv_free, kCompThreads);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, Ly::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // From here on the kernel reads what earlier work on the stream wrote.
  griddep_wait();
  griddep_launch_dependents();

  // ---- Q tile -> f16 (all threads), K-major SW128 ----
  {
    uint8_t* q16 = smem + Ly::oQ;
    constexpr int CH = D / 16;  // int8 chunks per row
    for (int i = tid; i < kRows * CH; i += kThreads) {
      const int rr = i / CH, dc = i % CH;
      const int r = r0 + rr;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < R) {
        const int j = r / G, hq = kvh * G + r % G;
        v = __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t)j * Hq + hq) * D) + dc);
      }
      uint4 h0, h1;
      s8x16_to_f16(v, h0, h1);
      uint8_t* atom = q16 + (size_t)(dc / 4) * (kRows * 128);
      *reinterpret_cast<uint4*>(atom + swz_chunk<128>(rr, 2 * (dc % 4))) = h0;
      *reinterpret_cast<uint4*>(atom + swz_chunk<128>(rr, 2 * (dc % 4) + 1)) = h1;
    }
    fence_async_smem();
  }
  __syncthreads();

  if (warp < kCompWarp0) {
    regs_dec<56>();  // warpgroup 0 hands registers to the softmax/output warpgroups
    if (warp != kMmaWarp) {
      // ================= copies and conversion (warps 0, 2, 3) =================
      const int ct = warp == 0 ? lane : tid - 32;  // 0 .. 95
      const uint32_t srow = kBS * Hkv * 4;
      auto issue = [&](int g) {  // warp 0 lane 0
        const int st = g % kStages;
        uint8_t* base = smem + Ly::oStage + (size_t)st * Ly::kStage;
        int blks[kPagesPG];
        int nb = 0;
#pragma unroll
        for (int i = 0; i < kPagesPG; ++i) {
          const int lb = g * kPagesPG + i;
          int blk = -1;
          if (lb < max_blk) {
            blk = p.block_table[lb];
            if (blk < 0 || blk >= p.num_blocks) {
              record_error(2);
              blk = -1;
            }
          }
          blks[i] = blk;
          nb += blk >= 0;
        }
        mbar_expect_tx(&stage_full[st], nb * (2 * Ly::kPage + 2 * srow));
#pragma unroll
        for (int i = 0; i < kPagesPG; ++i) {
          if (blks[i] < 0) continue;
          const size_t page = ((size_t)blks[i] * Hkv + kvh) * Ly::kPage;
          bulk_g2s(base + i * Ly::kPage, p.k_cache + page, Ly::kPage, &stage_full[st]);
          bulk_g2s(base + (kPagesPG + i) * Ly::kPage, p.v_cache + page, Ly::kPage, &stage_full[st]);
          const size_t so = (size_t)blks[i] * kBS * Hkv;
          bulk_g2s(base + 2 * kPagesPG * Ly::kPage + i * Ly::kSRow, p.k_scale + so, srow, &stage_full[st]);
          bulk_g2s(base + 2 * kPagesPG * Ly::kPage + (kPagesPG + i) * Ly::kSRow, p.v_scale + so, srow,
                   &stage_full[st]);
        }
        mbar_arrive(&stage_full[st]);
      };
      int issued = 0;  // groups whose copies were issued (warp 0 lane 0)
      if (warp == 0 && lane == 0)
        for (; issued < kStages && issued < ng; ++issued) issue(issued);
      for (int g = 0; g < ng; ++g) {
        const int st = g % kStages, sl = g & 1;
        pwait(&stage_full[st], (g / kStages) & 1, abort_flag);
        if (g >= 2) pwait(&mma_done[sl], ((g - 2) >> 1) & 1, abort_flag);  // PV(g-2) has read the slot
        const uint8_t* kt = smem + Ly::oStage + (size_t)st * Ly::kStage;
        const uint8_t* vt = kt + kPagesPG * Ly::kPage;
        const float* sks = reinterpret_cast<const float*>(kt + 2 * kPagesPG * Ly::kPage);
        const float* svs = sks + kPagesPG * Ly::kSRow / 4;
        uint8_t* k16 = smem + Ly::oK + (size_t)sl * Ly::kK16;
        uint8_t* v16 = smem + Ly::oV + (size_t)sl * Ly::kV16;
        // K page [D/16][16 tokens][16 B] -> [key][D]: chunk i = (page, dim chunk, token)
        constexpr int KC = kPagesPG * (D / 16) * kBS;
        for (int i = ct; i < KC; i += kConvThreads) {
          const int pg = i / ((D / 16) * kBS), rem = i % ((D / 16) * kBS);
          const int dc = rem / kBS, tk = rem % kBS;
          const uint4 v = *reinterpret_cast<const uint4*>(kt + (size_t)pg * Ly::kPage + (size_t)rem * 16);
          uint4 h0, h1;
          s8x16_to_f16(v, h0, h1);
          const int key = pg * kBS + tk;
          uint8_t* atom = k16 + (size_t)(dc / 4) * (kGroup * 128);
          *reinterpret_cast<uint4*>(atom + swz_chunk<128>(key, 2 * (dc % 4))) = h0;
          *reinterpret_cast<uint4*>(atom + swz_chunk<128>(key, 2 * (dc % 4) + 1)) = h1;
        }
        // V page [D][16 tokens] -> [D][32 keys]: chunk i = (page, dim)
        for (int i = ct; i < kPagesPG * D; i += kConvThreads) {
          const int pg = i / D, d = i % D;
          const uint4 v = *reinterpret_cast<const uint4*>(vt + (size_t)pg * Ly::kPage + (size_t)d * 16);
          uint4 h0, h1;
          s8x16_to_f16(v, h0, h1);
          *reinterpret_cast<uint4*>(v16 + swz_chunk<64>(d, 2 * pg)) = h0;
          *reinterpret_cast<uint4*>(v16 + swz_chunk<64>(d, 2 * pg + 1)) = h1;
        }
        if (ct < kGroup) {
          float2* sc = reinterpret_cast<float2*>(smem + Ly::oSc) + sl * kGroup;
          const int pg = ct / kBS, tk = ct % kBS;
          sc[ct] = make_float2(sks[pg * (Ly::kSRow / 4) + tk * Hkv + kvh], svs[pg * (Ly::kSRow / 4) + tk * Hkv + kvh]);
        }
        fence_async_smem();
        mbar_arrive(&conv_full[sl]);
        named_bar_sync(5, kConvThreads);  // every converter is done with staging buffer st
        if (warp == 0 && lane == 0 && issued < ng && !*abort_flag) issue(issued++);
      }
      if (warp == 0 && lane == 0) {
        // copies issued but never waited for (after an abort) land before the CTA exits
        for (int g = max(0, issued - kStages); g < issued; ++g) mbar_wait(&stage_full[g % kStages], (g / kStages) & 1);
      }
    } else {
      // ================= MMA issue (warp 1, lane 0) =================
      if (lane == 0) {
        constexpr uint32_t idesc_qk = umma_idesc_f16(kRows, kGroup);
        constexpr uint32_t idesc_pv = umma_idesc_f16(kRows, D);
        const uint32_t q16 = smem_u32(smem + Ly::oQ);
        for (int g = 0; g <= ng; ++g) {
          if (g < ng) {
            const int sl = g & 1;
            pwait(&conv_full[sl], (g >> 1) & 1, abort_flag);
            if (g >= 2) pwait(&s_free[sl], ((g - 2) >> 1) & 1, abort_flag);
            tc_fence_after();
            const uint32_t k16 = smem_u32(smem + Ly::oK + (size_t)sl * Ly::kK16);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t a = q16 + (kk / 4) * (kRows * 128) + (kk % 4) * 32;
              const uint32_t b = k16 + (kk / 4) * (kGroup * 128) + (kk % 4) * 32;
              umma_f16(tmem + 32 * sl, umma_desc(a, 128), umma_desc(b, 128), idesc_qk, kk > 0);
            }
            umma_commit(&s_full[sl]);
          }
          if (g >= 1) {
            const int h = g - 1, sl = h & 1;
            pwait(&p_full[sl], (h >> 1) & 1, abort_flag);
            if (h >= 1) pwait(pv_free, (h - 1) & 1, abort_flag);
            tc_fence_after();
            const uint32_t p16 = smem_u32(smem + Ly::oP + (size_t)sl * Ly::kP16);
            const uint32_t v16 = smem_u32(smem + Ly::oV + (size_t)sl * Ly::kV16);
#pragma unroll
            for (int kk = 0; kk < kGroup / 16; ++kk)
              umma_f16(tmem + Ly::kPVCol, umma_desc(p16 + kk * 32, 64), umma_desc(v16 + kk * 32, 64), idesc_pv,
                       kk > 0);
            umma_commit(&mma_done[sl]);
          }
        }
        // every MMA has completed before TMEM is released (the last commit covers all)
        if (ng >= 1) mbar_wait(&mma_done[(ng - 1) & 1], ((ng - 1) >> 1) & 1);
      }
      __syncwarp();
    }
  } else {
    // ================= softmax and output (warps 4..11) =================
    regs_inc<216>();
    const int half = (warp - kCompWarp0) >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int r = r0 + row;
    const bool valid = r < R;
    const int j = valid ? r / G : 0, hq = kvh * G + (valid ? r % G : 0);
    const int lim = valid ? H + j : -1;  // last visible key
    const float sq = valid ? p.q_scale[(size_t)j * Hq + hq] : 0.f;
    const float csc = p.sm_scale;
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    const int pair_bar = 1 + quarter;  // named barrier of warps quarter + 4 and quarter + 8
    float* xm = xch;                   // [half][row] group maxima
    float* xa = xch + 2 * kRows;       // [half][row] group absmax of W
    float* xl = xch + 4 * kRows;       // [half][row] final row sums
    float o[DH];
#pragma unroll
    for (int i = 0; i < DH; ++i) o[i] = 0.f;
    float m = -INFINITY, l = 0.f;
    float prev_alpha = 1.f, prev_sw = 0.f;

    // o = alpha o + sW (Wq x Vq) of group h, read from TMEM
    auto update = [&](int h, float alpha, float sw) {
      pwait(&mma_done[h & 1], (h >> 1) & 1, abort_flag);
      tc_fence_after();
      const bool rescale = __any_sync(0xffffffffu, alpha != 1.f);
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
        float v[32];
        tmem_ld32(trow + Ly::kPVCol + half * DH + 32 * c, v);
        tmem_wait_ld();
        if (c == DH / 32 - 1) {
          tc_fence_before();
          mbar_arrive(pv_free);
        }
        if (rescale) {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[32 * c + i] = __fmaf_rn(v[i], sw, __fmul_rn(o[32 * c + i], alpha));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[32 * c + i] = __fmaf_rn(v[i], sw, o[32 * c + i]);
        }
      }
    };

    for (int g = 0; g < ng; ++g) {
      const int sl = g & 1;
      pwait(&s_full[sl], (g >> 1) & 1, abort_flag);
      tc_fence_after();
      float s[16];
      tmem_ld16(trow + 32 * sl + 16 * half, s);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&s_free[sl]);
      pwait(&conv_full[sl], (g >> 1) & 1, abort_flag);  // the group's scales (already complete)
      const float4* sc4 = reinterpret_cast<const float4*>(smem + Ly::oSc) + sl * (kGroup / 2) + half * 8;
      float sk[16], sv[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 f = sc4[i];
        sk[2 * i] = f.x;
        sv[2 * i] = f.y;
        sk[2 * i + 1] = f.z;
        sv[2 * i + 1] = f.w;
      }
      // ---- scores (acc x sQ x sK x scale), causal mask, the group's row maximum ----
      const int key0 = g * kGroup + half * 16;
      float gmh = -INFINITY;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        s[i] = key0 + i <= lim ? __fmul_rn(__fmul_rn(__fmul_rn(s[i], sq), sk[i]), csc) : -INFINITY;
        gmh = fmaxf(gmh, s[i]);
      }
      xm[half * kRows + row] = gmh;
      named_bar_sync(pair_bar, 64);
      const float gm = fmaxf(xm[row], xm[kRows + row]);
      // ---- online softmax: m' = max(m, gm), alpha = exp(m - m'), p~ = exp(s - m') ----
      const float mn = fmaxf(m, gm);
      float alpha = 1.f;
      float w[16];
      float ah = 0.f, lsum = 0.f;
      if (mn != -INFINITY) {
        alpha = m == -INFINITY ? 0.f : expf(__fsub_rn(m, mn));
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float pe = expf(__fsub_rn(s[i], mn));  // 0 for masked keys
          lsum += pe;
          w[i] = pe != 0.f ? __fmul_rn(pe, sv[i]) : 0.f;
          ah = fmaxf(ah, w[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = 0.f;
      }
      m = mn;
      l = __fmaf_rn(l, alpha, lsum);
      xa[half * kRows + row] = ah;
      named_bar_sync(pair_bar, 64);
      const float A = fmaxf(xa[row], xa[kRows + row]);
      // sW = A / 127 and the codes round(W / sW), both IEEE fp32 quotients (W / sW
      // by Markstein's method); W / sW <= A / RN(A / 127) < 127.5, no clamp needed
      const float sw = div127(A);
      const float ysw = __frcp_rn(sw);
      const bool tiny = sw < kTinyDivisor;
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float c0 = A > 0.f ? rintf(div_shared(w[2 * i], sw, ysw, tiny)) : 0.f;
        const float c1 = A > 0.f ? rintf(div_shared(w[2 * i + 1], sw, ysw, tiny)) : 0.f;
        pk[i] = f16x2_of(c0, c1);
      }
      // ---- Wq (f16) -> the PV A tile: row `row`, keys 16 half .. 16 half + 15 ----
      if (g >= 2) pwait(&mma_done[sl], ((g - 2) >> 1) & 1, abort_flag);  // PV(g-2) has read the slot
      uint8_t* p16 = smem + Ly::oP + (size_t)sl * Ly::kP16;
      *reinterpret_cast<uint4*>(p16 + swz_chunk<64>(row, 2 * half)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      *reinterpret_cast<uint4*>(p16 + swz_chunk<64>(row, 2 * half + 1)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      fence_async_smem();
      mbar_arrive(&p_full[sl]);
      // ---- the previous group's product joins the output ----
      if (g >= 1) update(g - 1, prev_alpha, prev_sw);
      prev_alpha = alpha;
      prev_sw = sw;
    }
    if (ng >= 1) update(ng - 1, prev_alpha, prev_sw);

    // ---- finish: O = o / l ----
    xl[half * kRows + row] = l;
    named_bar_sync(pair_bar, 64);
    const float lt = xl[row] + xl[kRows + row];
    if (valid) {
      const float inv = 1.0f / lt;
      float4* orow = reinterpret_cast<float4*>(p.out + ((size_t)j * Hq + hq) * D + half * DH);
#pragma unroll
      for (int i = 0; i < DH / 4; ++i)
        orow[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, Ly::kTmemCols);
  }
}

}  // namespace

cudaError_t launch_int8_prefix(const PrefixParams& p, cudaStream_t stream) {
  const int R = p.C * p.G;
  dim3 grid((R + kRows - 1) / kRows, p.Hkv);
  cudaError_t e;
  if (p.D == 256) {
    e = cudaFuncSetAttribute(int8_prefix_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay<256>::kTotal);
    if (e != cudaSuccess) return e;
    return launch_pdl(int8_prefix_kernel<256>, grid, dim3(kThreads), Lay<256>::kTotal, stream, p);
  }
  e = cudaFuncSetAttribute(int8_prefix_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay<128>::kTotal);
  if (e != cudaSuccess) return e;
  return launch_pdl(int8_prefix_kernel<128>, grid, dim3(kThreads), Lay<128>::kTotal, stream, p);
}

}  // namespace i8kv
