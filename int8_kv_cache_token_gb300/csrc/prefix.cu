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
// GB300 shape.  A CTA owns 128 query rows of one KV head (8 warps x 16 rows);
// the rows are (chunk token, query head) pairs of that KV head's GQA group,
// token-major, so the query heads sharing K/V read the same tiles.  K/V pages
// of 64 keys per stage arrive by bulk copy into a double-buffered int8 staging
// area.  Each stage is then converted once, by all warps together, into f16
// tiles in shared memory: K as [key][dim] and V as [dim][key], 16-byte chunks
// XOR-swizzled so that ldmatrix reads them without bank conflicts.  The int8
// values are exact in f16, every product is exact and every partial sum stays
// below 2^22, so the f16 tensor-core MMAs with fp32 accumulation give the exact
// int32 results of the INT8 contractions (QK over D dims; PV over one 32-key
// group).  Each warp keeps its rows' softmax state and FP32 output in registers
// (FlashAttention-2 style).  Per 32-key group: QK, scores, causal mask, online
// softmax, W = p~ x sV, per-row group absmax, sW = A / 127 and the codes
// round(W / sW) (IEEE quotients, as the oracle), then PV with the codes as the
// A operand and sW x (the exact product) added to the output.
#include "common.cuh"
#include "kernels.h"

namespace i8kv {
I8KV_DEFINE_ERROR_ACCESSOR(read_error_prefix)

namespace {

constexpr int kBS = 16;
constexpr int kWarps = 8;
constexpr int kRowsPerCTA = kWarps * 16;
constexpr int kKeysPerStage = 64;  // 4 blocks
constexpr int kBlocksPerStage = kKeysPerStage / kBS;
constexpr int kStages = 2;         // int8 staging buffers
constexpr int kMaxHkv = 8;

template <int D>
struct PrefixSmem {
  static constexpr int kPage = D * kBS;                           // int8 page
  static constexpr int kTileBytes = kBlocksPerStage * kPage;      // int8 K (or V) tile of a stage
  static constexpr int kScaleBytes = kBlocksPerStage * kBS * kMaxHkv * 4;
  static constexpr int kStageBytes = 2 * kTileBytes + 2 * kScaleBytes;
  static constexpr int kK16 = kKeysPerStage * D * 2;              // f16 K [64 keys][D]
  static constexpr int kV16 = D * kKeysPerStage * 2;              // f16 V [D][64 keys]
  static constexpr int kQ16 = kRowsPerCTA * D * 2;                // f16 Q [128 rows][D]
  static constexpr int kSc = kKeysPerStage * 2 * 4;               // the stage's (sK, sV) per key
  static constexpr int kOffK16 = kStages * kStageBytes;
  static constexpr int kOffV16 = kOffK16 + kK16;
  static constexpr int kOffQ16 = kOffV16 + kV16;
  static constexpr int kOffSc = kOffQ16 + kQ16;
  static constexpr int kOffBar = kOffSc + kSc;
  static constexpr int kTotal = kOffBar + 64;
};

// 16 int8 codes (one 16-byte chunk) -> 16 exact f16 values, natural order.
__device__ __forceinline__ void s8x16_to_f16(const uint4& v, uint4& h0, uint4& h1) {
  s8x4_to_f16(v.x, h0.x, h0.y);
  s8x4_to_f16(v.y, h0.z, h0.w);
  s8x4_to_f16(v.z, h1.x, h1.y);
  s8x4_to_f16(v.w, h1.z, h1.w);
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32, 1) int8_prefix_kernel(PrefixParams p) {
  using S = PrefixSmem<D>;
  constexpr int KS = D / 16;  // k16 steps of QK
  constexpr int ND = D / 8;   // n-tiles of PV
  constexpr int KC = (D / 16) * kBS;  // int8 chunks of one K page
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* k16 = smem + S::kOffK16;
  uint8_t* v16 = smem + S::kOffV16;
  uint8_t* q16 = smem + S::kOffQ16;
  float* scs = reinterpret_cast<float*>(smem + S::kOffSc);  // [64 keys][sK, sV]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + kStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int kvh = blockIdx.y;
  const int G = p.G, Hkv = p.Hkv, Hq = p.Hq, H = p.H, C = p.C;
  const int R = C * G;
  // Row blocks in reverse: later chunk tokens see more keys, and CTAs start in
  // index order, so the heaviest blocks run first and the partial last wave
  // holds the lightest ones.
  const int r0 = (gridDim.x - 1 - blockIdx.x) * kRowsPerCTA;
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

  // ---- query tile -> shared memory as exact f16, natural dim order; 16-byte
  // chunk c of row r is stored at chunk c ^ (r & 7) ----
  for (int i = tid; i < kRowsPerCTA * (D / 16); i += kWarps * 32) {
    const int rr = i / (D / 16), c16 = i % (D / 16);
    const int r = r0 + rr;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < R) {
      const int j = r / G, hq = kvh * G + r % G;
      v = __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t)j * Hq + hq) * D) + c16);
    }
    uint4 h0, h1;
    s8x16_to_f16(v, h0, h1);
    uint8_t* row = q16 + (size_t)rr * (2 * D);
    *reinterpret_cast<uint4*>(row + (((2 * c16) ^ (rr & 7)) * 16)) = h0;
    *reinterpret_cast<uint4*>(row + (((2 * c16 + 1) ^ (rr & 7)) * 16)) = h1;
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
    __syncthreads();  // every warp is done with the previous stage's f16 tiles
    // ---- convert the stage once: int8 pages -> f16 tiles, scales -> scs ----
    {
      const uint8_t* kt = stage_base(b);
      const uint8_t* vt = kt + S::kTileBytes;
      const float* sks = reinterpret_cast<const float*>(kt + 2 * S::kTileBytes);
      const float* svs = sks + S::kScaleBytes / 4;
      // K page [D/16][16 tokens][16 B] -> K16 [key][D]
      for (int i = tid; i < kBlocksPerStage * KC; i += kWarps * 32) {
        const int pg = i / KC, rem = i % KC;
        const int c16 = rem / kBS, tk = rem % kBS;
        const uint4 v = *reinterpret_cast<const uint4*>(kt + (size_t)pg * S::kPage + (size_t)rem * 16);
        const int key = pg * kBS + tk;
        uint4 h0, h1;
        s8x16_to_f16(v, h0, h1);
        uint8_t* row = k16 + (size_t)key * (2 * D);
        *reinterpret_cast<uint4*>(row + (((2 * c16) ^ (key & 7)) * 16)) = h0;
        *reinterpret_cast<uint4*>(row + (((2 * c16 + 1) ^ (key & 7)) * 16)) = h1;
      }
      // V page [D][16 tokens] -> V16 [D][64 keys]
      for (int i = tid; i < kBlocksPerStage * D; i += kWarps * 32) {
        const int pg = i / D, d = i % D;
        const uint4 v = *reinterpret_cast<const uint4*>(vt + (size_t)pg * S::kPage + (size_t)d * 16);
        uint4 h0, h1;
        s8x16_to_f16(v, h0, h1);
        uint8_t* row = v16 + (size_t)d * (2 * kKeysPerStage);
        *reinterpret_cast<uint4*>(row + (((2 * pg) ^ (d & 7)) * 16)) = h0;
        *reinterpret_cast<uint4*>(row + (((2 * pg + 1) ^ (d & 7)) * 16)) = h1;
      }
      if (tid < kKeysPerStage) {
        scs[2 * tid] = sks[tid * Hkv + kvh];
        scs[2 * tid + 1] = svs[tid * Hkv + kvh];
      }
    }
    __syncthreads();  // the f16 tiles are ready; the int8 buffer b is free
    if (tid == 0 && st + kStages < n_stages) issue(st + kStages);

#pragma unroll 1
    for (int grp = 0; grp < kKeysPerStage / 32; ++grp) {
      const int key0 = st * kKeysPerStage + grp * 32;  // absolute position of the group's first key
      if (key0 > warp_lim) break;                       // every row of this warp is past its causal limit
      // ---- QK: 4 n-tiles of 8 keys, exact on the f16 tensor path ----
      float acc[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
      {
        // A (query rows): matrices (rows 0-7 | 8-15) x (dim chunk 2kk | 2kk+1)
        const int qr = warp * 16 + ri + 8 * (mi & 1);
        const uint8_t* qrow = q16 + (size_t)qr * (2 * D);
        // B (keys): matrices (n-tile 2np2 | 2np2+1) x (dim chunk 2kk | 2kk+1)
        const uint8_t* krow[2];
        int kxor[2];
#pragma unroll
        for (int np2 = 0; np2 < 2; ++np2) {
          const int key = grp * 32 + 8 * (2 * np2 + (mi >> 1)) + ri;  // key within the stage
          krow[np2] = k16 + (size_t)key * (2 * D);
          kxor[np2] = key & 7;
        }
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t a[4];
          ldmatrix_x4(a, qrow + (((2 * kk + (mi >> 1)) ^ (qr & 7)) * 16));
#pragma unroll
          for (int np2 = 0; np2 < 2; ++np2) {
            uint32_t bb[4];
            ldmatrix_x4(bb, krow[np2] + (((2 * kk + (mi & 1)) ^ kxor[np2]) * 16));
            mma_f16_16816(acc[2 * np2], a[0], a[1], a[2], a[3], bb[0], bb[1]);
            mma_f16_16816(acc[2 * np2 + 1], a[0], a[1], a[2], a[3], bb[2], bb[3]);
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
          const int kl = grp * 32 + 8 * n + 2 * t + (e & 1);  // key within the stage
          const int key = st * kKeysPerStage + kl;
          const int h2 = e >> 1;
          float s = -INFINITY;
          if (key <= row_lim[h2] && key < total_keys)
            s = __fmul_rn(__fmul_rn(__fmul_rn(acc[n][e], sq[h2]), scs[2 * kl]), csc);
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
            we = __fmul_rn(pe, scs[2 * (grp * 32 + 8 * n + 2 * t + (e & 1)) + 1]);
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
        sW[h2] = div127(A[h2]);
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
      // A operand of PV (exact integers in f16): k16 step kk covers the group's
      // keys 16kk .. 16kk+15 = score n-tiles 2kk (a0: row g, a1: row g+8) and
      // 2kk+1 (a2, a3).
      uint32_t pa[2][4];
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        pa[kk][0] = f16x2_of(q[2 * kk][0], q[2 * kk][1]);
        pa[kk][1] = f16x2_of(q[2 * kk][2], q[2 * kk][3]);
        pa[kk][2] = f16x2_of(q[2 * kk + 1][0], q[2 * kk + 1][1]);
        pa[kk][3] = f16x2_of(q[2 * kk + 1][2], q[2 * kk + 1][3]);
      }
      if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
        for (int n = 0; n < ND; ++n) {
          o[n][0] *= alpha[0];
          o[n][1] *= alpha[0];
          o[n][2] *= alpha[1];
          o[n][3] *= alpha[1];
        }
      }
      // ---- PV: B = V tile [dim][key]: matrices (dim n-tile dn | dn+1) x (key chunk c | c+1) ----
#pragma unroll
      for (int dn = 0; dn < ND; dn += 2) {
        const int d = 8 * (dn + (mi >> 1)) + ri;
        const uint8_t* vrow = v16 + (size_t)d * (2 * kKeysPerStage);
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int chunk = 4 * grp + 2 * kk + (mi & 1);
          uint32_t bb[4];
          ldmatrix_x4(bb, vrow + ((chunk ^ (d & 7)) * 16));
          mma_f16_16816(c0, pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], bb[0], bb[1]);
          mma_f16_16816(c1, pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], bb[2], bb[3]);
        }
        o[dn][0] = fmaf(c0[0], sW[0], o[dn][0]);
        o[dn][1] = fmaf(c0[1], sW[0], o[dn][1]);
        o[dn][2] = fmaf(c0[2], sW[1], o[dn][2]);
        o[dn][3] = fmaf(c0[3], sW[1], o[dn][3]);
        o[dn + 1][0] = fmaf(c1[0], sW[0], o[dn + 1][0]);
        o[dn + 1][1] = fmaf(c1[1], sW[0], o[dn + 1][1]);
        o[dn + 1][2] = fmaf(c1[2], sW[1], o[dn + 1][2]);
        o[dn + 1][3] = fmaf(c1[3], sW[1], o[dn + 1][3]);
      }
    }
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
