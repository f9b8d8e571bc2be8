// prefix.cu -- INT8 prefix-prefill chunk attention.
//
// Source: "gfx936 DCU上实现INT8 PV MMAC：V Scale融合、概率量化与Fragment分组"
// §2.1 (the prefix keeps one online softmax (m, l, o); alpha = exp(m - m'),
// p~ = exp(score - m'), W = p~ x sV is quantized unnormalized; O = o / l at
// the end), §1 and §3 (32-token probability groups, sW = max W / 127, W on the
// A side and V on the B side of the INT8 MMA) and "gfx936 DCU上实现INT8 KV与
// INT8 MMAC Attention推理优化" §3.2 (history and the chunk's own K/V in one
// online softmax, never two attentions merged afterwards).
//
// GB300 shape.  A CTA owns 64 query rows of one KV head (4 warps x 16 rows);
// the rows are (chunk token, query head) pairs of that KV head's GQA group,
// token-major, so the 6 query heads sharing K/V read the same shared-memory
// tiles.  K/V pages of 64 keys per stage arrive by bulk copy (thread 0 issues,
// mbarrier completes), double-buffered.  Each warp keeps its rows' softmax
// state and the FP32 output in registers (FlashAttention-2 style).  Per
// 32-key group: QK with mma.sync m16n8k32 s8 whose B fragments are loaded with
// a key order permuted inside the group, so the score fragments land exactly
// where the PV A operand needs the 32 codes of the group (the group's set of
// tokens is unchanged; only the order inside the MMA's K dimension differs);
// then scores, causal mask, online softmax, W = p~ x sV, per-row group absmax,
// quantize, and PV with mma.sync s8 (B = V pages via ldmatrix), the int32
// result scaled by the row's sW into the FP32 accumulators.
#include "common.cuh"
#include "kernels.h"

namespace i8kv {
I8KV_DEFINE_ERROR_ACCESSOR(read_error_prefix)

namespace {

constexpr int kBS = 16;
constexpr int kRowsPerCTA = 64;
constexpr int kWarps = 4;
constexpr int kKeysPerStage = 64;  // 4 blocks
constexpr int kBlocksPerStage = kKeysPerStage / kBS;
constexpr int kStages = 2;

template <int D>
struct PrefixSmem {
  static constexpr int kPage = D * kBS;
  static constexpr int kTileBytes = kBlocksPerStage * kPage;
  // per stage: K tile, V tile, K-scale rows, V-scale rows (Hkv <= 8)
  static constexpr int kScaleBytes = kBlocksPerStage * kBS * 8 * 4;
  static constexpr int kStageBytes = 2 * kTileBytes + 2 * kScaleBytes;
  static constexpr int kQBytes = kRowsPerCTA * D * 2;  // f16 query tile, 16-byte chunks XOR-swizzled by row
  static constexpr int kTotal = kStages * kStageBytes + kQBytes + 64;
};

// Key offset (within a 32-key group) of column c of QK n-tile nn (0..3).
__device__ __forceinline__ int group_key(int nn, int c) {
  const int base = (nn & 1) * 2 + (nn >> 1) * 16;
  return base + 4 * (c >> 1) + (c & 1);
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) int8_prefix_kernel(PrefixParams p) {
  using S = PrefixSmem<D>;
  constexpr int KS = D / 32;  // k-steps of QK
  constexpr int ND = D / 8;   // n-tiles of PV
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* qs = smem + kStages * S::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * S::kStageBytes + S::kQBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + kStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int kvh = blockIdx.y;
  const int G = p.G, Hkv = p.Hkv, Hq = p.Hq, H = p.H, C = p.C;
  const int R = C * G;
  const int r0 = blockIdx.x * kRowsPerCTA;
  const int total_keys = H + C;
  const int j_hi = min(C - 1, (r0 + kRowsPerCTA - 1) / G);
  const int n_keys = H + j_hi + 1;
  const int n_stages = (n_keys + kKeysPerStage - 1) / kKeysPerStage;
  const int max_blk = (total_keys + kBS - 1) / kBS;

  auto stage_base = [&](int b) { return smem + (size_t)b * S::kStageBytes; };
  auto issue = [&](int st) {
    const int b = st % kStages;
    uint8_t* base = stage_base(b);
    int nb = 0;
    int blks[kBlocksPerStage];
#pragma unroll
    for (int i = 0; i < kBlocksPerStage; ++i) {
      const int lb = st * kBlocksPerStage + i;
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
    const uint32_t srow = kBS * Hkv * 4;
    mbar_expect_tx(&full[b], nb * (2 * S::kPage + 2 * srow));
#pragma unroll
    for (int i = 0; i < kBlocksPerStage; ++i) {
      if (blks[i] < 0) continue;
      const size_t page = ((size_t)blks[i] * Hkv + kvh) * S::kPage;
      bulk_g2s(base + i * S::kPage, p.k_cache + page, S::kPage, &full[b]);
      bulk_g2s(base + S::kTileBytes + i * S::kPage, p.v_cache + page, S::kPage, &full[b]);
      bulk_g2s(base + 2 * S::kTileBytes + i * srow, p.k_scale + (size_t)blks[i] * kBS * Hkv, srow, &full[b]);
      bulk_g2s(base + 2 * S::kTileBytes + S::kScaleBytes + i * srow, p.v_scale + (size_t)blks[i] * kBS * Hkv, srow,
               &full[b]);
    }
    mbar_arrive(&full[b]);
  };

  if (tid == 0) {
    for (int b = 0; b < kStages; ++b) mbar_init(&full[b], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int st = 0; st < kStages && st < n_stages; ++st) issue(st);
  }

  // ---- query tile -> shared memory as exact f16 ----
  // Head-dims are stored in the order the k16 MMAs consume them next to K
  // fragments converted by s8b_to_f16: inside each 16-dim half of a 32-dim
  // step, logical positions 0..7 hold physical dims {0,1,4,5,8,9,12,13} and
  // 8..15 hold {2,3,6,7,10,11,14,15}.  Logical 16-byte chunk c (8 f16) of row r
  // is stored at chunk c ^ (r & 7).
  for (int i = tid; i < kRowsPerCTA * (D / 8); i += kWarps * 32) {
    const int rr = i / (D / 8), ch = i % (D / 8);
    const int r = r0 + rr;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < R) {
      const int j = r / G, hq = kvh * G + r % G;
      v = __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t)j * Hq + hq) * D) + (ch >> 1));
    }
    const uint32_t sel = (ch & 1) ? 0x7632u : 0x5410u;
    const uint32_t x0 = __byte_perm(v.x, v.y, sel), x1 = __byte_perm(v.z, v.w, sel);
    uint4 h;
    s8x4_to_f16(x0, h.x, h.y);
    s8x4_to_f16(x1, h.z, h.w);
    *reinterpret_cast<uint4*>(qs + (size_t)rr * (2 * D) + ((ch ^ (rr & 7)) * 16)) = h;
  }
  // ---- this warp's 16 rows: (token, head), causal limit, query scale ----
  int row_lim[2];
  float sq[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int r = r0 + warp * 16 + g + 8 * h2;
    const bool ok = r < R;
    const int j = ok ? r / G : C - 1;
    const int hq = kvh * G + (ok ? r % G : 0);
    row_lim[h2] = H + j;  // last visible key
    sq[h2] = ok ? p.q_scale[(size_t)j * Hq + hq] : 0.f;
  }
  const int warp_lim = __shfl_sync(0xffffffffu, row_lim[1], 31);  // rows are token-major: last row sees most
  __syncthreads();

  float o[ND][4];
#pragma unroll
  for (int n = 0; n < ND; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  const float csc = p.sm_scale;
  const int mi = lane >> 3, ri = lane & 7;

  for (int st = 0; st < n_stages; ++st) {
    const int b = st % kStages;
    // bounded wait (see common.cuh); every thread passes the same barriers
    if (!mbar_try_wait(&full[b], (st / kStages) & 1)) {
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&full[b], (st / kStages) & 1)) {
        if (*abort_flag) break;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          record_error(1);
          *abort_flag = 1;
          break;
        }
      }
    }
    const int8_t* kt = reinterpret_cast<const int8_t*>(stage_base(b));
    const int8_t* vt = kt + S::kTileBytes;
    const float* sks = reinterpret_cast<const float*>(kt + 2 * S::kTileBytes);
    const float* svs = sks + S::kScaleBytes / 4;
#pragma unroll 1
    for (int grp = 0; grp < kKeysPerStage / 32; ++grp) {
      const int key0 = st * kKeysPerStage + grp * 32;  // absolute position of the group's first key
      if (key0 > warp_lim) break;                       // every row of this warp is past its causal limit
      // ---- QK: 4 n-tiles of 8 permuted keys, exact on the f16 tensor path ----
      float acc[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
      {
        // A (query rows, f16): matrices (rows 0-7 | 8-15) x (logical chunk c | c+1)
        const int qr = warp * 16 + ri + 8 * (mi & 1);
        const uint8_t* qrow = qs + (size_t)qr * (2 * D);
        // B (keys, s8): lanes 0-7 n-tile 2*np2 chunk 2s, 8-15 chunk 2s+1, 16-31 n-tile 2*np2+1
        const int8_t* krow[2];
#pragma unroll
        for (int np2 = 0; np2 < 2; ++np2) {
          const int kl = grp * 32 + group_key(2 * np2 + (mi >> 1), ri);  // key within the stage
          krow[np2] = kt + (kl >> 4) * S::kPage + (kl & 15) * 16 + (mi & 1) * (kBS * 16);
        }
#pragma unroll
        for (int s = 0; s < KS; ++s) {
          uint32_t a1[4], a2[4];
          ldmatrix_x4(a1, qrow + (((4 * s + (mi >> 1)) ^ (qr & 7)) * 16));
          ldmatrix_x4(a2, qrow + (((4 * s + 2 + (mi >> 1)) ^ (qr & 7)) * 16));
#pragma unroll
          for (int np2 = 0; np2 < 2; ++np2) {
            uint32_t bb[4], f0[4], f1[4];
            ldmatrix_x4(bb, krow[np2] + (size_t)(2 * s) * (kBS * 16));
            s8b_to_f16(bb[0], bb[1], f0);
            s8b_to_f16(bb[2], bb[3], f1);
            mma_f16_16816(acc[2 * np2], a1[0], a1[1], a1[2], a1[3], f0[0], f0[1]);
            mma_f16_16816(acc[2 * np2], a2[0], a2[1], a2[2], a2[3], f0[2], f0[3]);
            mma_f16_16816(acc[2 * np2 + 1], a1[0], a1[1], a1[2], a1[3], f1[0], f1[1]);
            mma_f16_16816(acc[2 * np2 + 1], a2[0], a2[1], a2[2], a2[3], f1[2], f1[3]);
          }
        }
      }
      // ---- scores, mask, online softmax ----
      float sc[4][4];
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kg = group_key(n, 2 * t + (e & 1));
          const int key = key0 + kg;
          const int h2 = e >> 1;
          float s = -INFINITY;
          if (key <= row_lim[h2] && key < total_keys) {
            const int kl = grp * 32 + kg;
            s = __fmul_rn(__fmul_rn(__fmul_rn(acc[n][e], sq[h2]), sks[kl * Hkv + kvh]), csc);
          }
          sc[n][e] = s;
          mx[h2] = fmaxf(mx[h2], s);
        }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 1));
        mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 2));
      }
      float alpha[2], mnew[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        mnew[h2] = fmaxf(m[h2], mx[h2]);
        alpha[h2] = (m[h2] == -INFINITY) ? 0.f : expf(m[h2] - mnew[h2]);
        m[h2] = mnew[h2];
        l[h2] *= alpha[h2];
      }
      float w[4][4];
      float A[2] = {0.f, 0.f};
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h2 = e >> 1;
          float pe = 0.f, we = 0.f;
          if (sc[n][e] != -INFINITY) {
            pe = expf(__fsub_rn(sc[n][e], mnew[h2]));
            const int kl = grp * 32 + group_key(n, 2 * t + (e & 1));
            we = __fmul_rn(pe, svs[kl * Hkv + kvh]);
          }
          l[h2] += pe;
          w[n][e] = we;
          A[h2] = fmaxf(A[h2], we);
        }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        A[h2] = fmaxf(A[h2], __shfl_xor_sync(0xffffffffu, A[h2], 1));
        A[h2] = fmaxf(A[h2], __shfl_xor_sync(0xffffffffu, A[h2], 2));
      }
      // sW = A / 127 and the codes round(W / sW), both IEEE fp32 quotients (W / sW
      // by Markstein's method); W / sW <= A / RN(A / 127) < 127.5, no clamp needed
      float sW[2], ysw[2];
      bool tiny[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        sW[h2] = __fdiv_rn(A[h2], 127.0f);
        ysw[h2] = __frcp_rn(sW[h2]);
        tiny[h2] = sW[h2] < kTinyDivisor;
      }
      float q[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h2 = e >> 1;
          q[n][e] = A[h2] > 0.f ? rintf(div_shared(w[n][e], sW[h2], ysw[h2], tiny[h2])) : 0.f;
        }
      // A operand of PV in f16 (exact integers): k16 MMA 1 takes the group's keys
      // 0..15, MMA 2 keys 16..31, with logical k (2t, 2t+1 | 2t+8, 2t+9) holding
      // keys (4t, 4t+1 | 4t+2, 4t+3) -- the order s8b_to_f16 gives the V fragments.
      uint32_t pa1[4], pa2[4];
      pa1[0] = f16x2_of(q[0][0], q[0][1]);
      pa1[1] = f16x2_of(q[0][2], q[0][3]);
      pa1[2] = f16x2_of(q[1][0], q[1][1]);
      pa1[3] = f16x2_of(q[1][2], q[1][3]);
      pa2[0] = f16x2_of(q[2][0], q[2][1]);
      pa2[1] = f16x2_of(q[2][2], q[2][3]);
      pa2[2] = f16x2_of(q[3][0], q[3][1]);
      pa2[3] = f16x2_of(q[3][2], q[3][3]);
      if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
        for (int n = 0; n < ND; ++n) {
          o[n][0] *= alpha[0];
          o[n][1] *= alpha[0];
          o[n][2] *= alpha[1];
          o[n][3] *= alpha[1];
        }
      }
      // ---- PV: B = V pages (rows = head-dims, 16 keys of one block per row) ----
      const int8_t* vb = vt + (size_t)(2 * grp + (mi & 1)) * S::kPage + ri * 16 + (mi >> 1) * (8 * 16);
#pragma unroll
      for (int n = 0; n < ND; n += 2) {
        uint32_t bb[4], f0[4], f1[4];
        ldmatrix_x4(bb, vb + (size_t)n * (8 * 16));
        s8b_to_f16(bb[0], bb[1], f0);
        s8b_to_f16(bb[2], bb[3], f1);
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16_16816(c0, pa1[0], pa1[1], pa1[2], pa1[3], f0[0], f0[1]);
        mma_f16_16816(c0, pa2[0], pa2[1], pa2[2], pa2[3], f0[2], f0[3]);
        mma_f16_16816(c1, pa1[0], pa1[1], pa1[2], pa1[3], f1[0], f1[1]);
        mma_f16_16816(c1, pa2[0], pa2[1], pa2[2], pa2[3], f1[2], f1[3]);
        o[n][0] += c0[0] * sW[0];
        o[n][1] += c0[1] * sW[0];
        o[n][2] += c0[2] * sW[1];
        o[n][3] += c0[3] * sW[1];
        o[n + 1][0] += c1[0] * sW[0];
        o[n + 1][1] += c1[1] * sW[0];
        o[n + 1][2] += c1[2] * sW[1];
        o[n + 1][3] += c1[3] * sW[1];
      }
    }
    __syncthreads();  // stage buffer b is free
    if (tid == 0 && st + kStages < n_stages) issue(st + kStages);
  }

  // ---- finish: O = o / l ----
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    l[h2] += __shfl_xor_sync(0xffffffffu, l[h2], 1);
    l[h2] += __shfl_xor_sync(0xffffffffu, l[h2], 2);
  }
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int r = r0 + warp * 16 + g + 8 * h2;
    if (r >= R) continue;
    const int j = r / G, hq = kvh * G + r % G;
    float* orow = p.out + ((size_t)j * Hq + hq) * D;
    const float inv = 1.0f / l[h2];
#pragma unroll
    for (int n = 0; n < ND; ++n) {
      float2 v2 = make_float2(o[n][2 * h2] * inv, o[n][2 * h2 + 1] * inv);
      *reinterpret_cast<float2*>(orow + 8 * n + 2 * t) = v2;
    }
  }
}

}  // namespace

cudaError_t launch_int8_prefix(const PrefixParams& p, cudaStream_t stream) {
  const int R = p.C * p.G;
  dim3 grid((R + kRowsPerCTA - 1) / kRowsPerCTA, p.Hkv);
  cudaError_t e;
  if (p.D == 256) {
    e = cudaFuncSetAttribute(int8_prefix_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PrefixSmem<256>::kTotal);
    if (e != cudaSuccess) return e;
    int8_prefix_kernel<256><<<grid, kWarps * 32, PrefixSmem<256>::kTotal, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(int8_prefix_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PrefixSmem<128>::kTotal);
    if (e != cudaSuccess) return e;
    int8_prefix_kernel<128><<<grid, kWarps * 32, PrefixSmem<128>::kTotal, stream>>>(p);
  }
  return cudaGetLastError();
}


}  // namespace i8kv
