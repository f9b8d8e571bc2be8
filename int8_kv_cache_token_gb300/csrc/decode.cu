// decode.cu -- INT8 paged decode attention (and the debug QK path).
//
// Source: "gfx936 DCU上实现INT8 PV MMAC：V Scale融合、概率量化与Fragment分组"
// §1 (W = P x sV, 32-token groups, sW = max W / 127), §2 (score recovery
// acc x sQ x sK / sqrt(d), online softmax), §2.2 (decode: 256-token partitions,
// P normalized inside the partition, log-sum-exp merge), §3 (P on the A side,
// V on the B side of the INT8 MMA; int32 bound 32 x 127 x 127 per group) and
// "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" §3.3 (the decode data
// flow) and §2.3 (cache layouts).
//
// GB300 design (not the pages' gfx936 one):
//  * Work unit = (sequence, KV head, 256-token partition).  A persistent grid of
//    one CTA per SM takes a contiguous range of units, so one CTA usually walks
//    several partitions of the same (sequence, KV head) and merges them
//    locally; pairs that span CTAs leave one partial per CTA in the workspace
//    and the last CTA to finish (an atomic ticket, no waiting) merges them.
//  * Warp 8 is a TMA producer: per unit it issues 16 bulk copies of K pages and
//    32 of scale rows (one item), then 16 of V pages (a second item), into a
//    ring of shared-memory slots guarded by full/empty mbarriers.
//  * Warps 0-7 consume.  GQA packs the G <= 8 query heads of one KV head into
//    the N = 8 side of mma.sync.m16n8k32 s8: QK has M = 16 tokens (one block),
//    K = 32 head-dims; PV has M = 16 head-dims, N = 8 query rows, K = the 32
//    tokens of one probability group, so every INT8 MMA consumes exactly one
//    aligned group and its scale sW is applied to that MMA's int32 result.
//  * Warp w computes QK, softmax terms and the W quantization of group w; the
//    quantized W fragments go through shared memory to all warps; warp w then
//    owns head-dims [w*D/8, (w+1)*D/8) of the PV output for the whole range.
#include "common.cuh"
#include "kernels.h"

namespace i8kv {

namespace {

constexpr int kPart = 256;   // partition (tokens) -- the pages' decode partition
constexpr int kBS = 16;      // block size
constexpr int kGroup = 32;   // probability group = K of one INT8 MMA
constexpr int kCWarps = 8;   // consumer warps (one per group of a partition)
constexpr int kThreads = (kCWarps + 1) * 32;
constexpr int kRows = 8;     // query rows in the MMA N dimension
constexpr int kWStride = 36; // padded row stride (floats) of the per-warp W staging
__host__ __device__ constexpr int kSlotFloats(int D) { return kRows * D + 2 * kRows; }

struct SmemLayout {
  int nslots, nsslots;
  size_t ring, scales, wbuf, wqf, swr, redmax, redsum, bars, ctrl, total;
};

__host__ __device__ inline SmemLayout decode_layout(int D, int Hkv, int nslots) {
  SmemLayout L;
  L.nslots = nslots;
  L.nsslots = (nslots + 2) / 2;
  const size_t item = (size_t)kPart * D;
  size_t off = 0;
  L.ring = off;
  off += (size_t)nslots * item;
  L.scales = off;
  off += (size_t)L.nsslots * 2 * kPart * Hkv * sizeof(float);
  L.wbuf = off;
  off += (size_t)kCWarps * kRows * kWStride * sizeof(float);
  L.wqf = off;
  off += (size_t)kCWarps * 32 * sizeof(uint2);
  L.swr = off;
  off += (size_t)kCWarps * kRows * sizeof(float);
  L.redmax = off;
  off += (size_t)kCWarps * kRows * sizeof(float);
  L.redsum = off;
  off += (size_t)kCWarps * kRows * sizeof(float);
  L.bars = off;
  off += (size_t)2 * nslots * sizeof(uint64_t);
  L.ctrl = off;
  off += 16 * sizeof(int);
  L.total = off;
  return L;
}

// Position in the (sequence, KV head, partition) unit order.
struct Walk {
  int b, kvh, part, L, np;
  long long ub;  // global index of the first unit of sequence b
};

__device__ __forceinline__ int clamp_len(int L, int maxL) {
  if (L < 0) return 0;
  return L > maxL ? maxL : L;
}

__device__ __forceinline__ void walk_next(Walk& w, const int32_t* seq_lens, int B, int Hkv, int maxL) {
  if (++w.part < w.np) return;
  w.part = 0;
  if (++w.kvh < Hkv) return;
  w.kvh = 0;
  w.ub += (long long)w.np * Hkv;
  for (;;) {
    if (++w.b >= B) return;
    w.L = clamp_len(seq_lens[w.b], maxL);
    w.np = (w.L + kPart - 1) / kPart;
    if (w.np > 0) return;
  }
}

// CTA whose unit range [c*U/N, (c+1)*U/N) holds unit u (N <= U: no empty ranges).
__device__ __forceinline__ int cta_of(long long u, long long U, int N) {
  return (int)(((u + 1) * N + U - 1) / U - 1);
}

// Bounded pipeline wait.  After a timeout (error 1) or once the CTA aborted,
// it returns without waiting so every thread still reaches the same barriers.
__device__ __forceinline__ void pipe_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return;
  if (*abort_flag) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      record_error(1);
      *abort_flag = 1;
      return;
    }
  }
}

// QK for the two 16-token blocks (2w, 2w+1) of a warp:
// acc[m][0..3] = (token g, row 2t), (token g, row 2t+1), (token g+8, row 2t), (token g+8, row 2t+1)
// of block 2w+m.  `kpages` holds 16 K pages [D/16][16 tokens][16 B].
template <int D>
__device__ __forceinline__ void qk_warp(const int8_t* kpages, int warp, int lane, const uint32_t (&qf)[D / 32][2],
                                        int (&acc)[2][4]) {
  const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
  for (int m = 0; m < 2; ++m) {
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[m][i] = 0;
    const int8_t* page = kpages + (size_t)(2 * warp + m) * (D * kBS);
    const int8_t* row = page + (mi >> 1) * (kBS * 16) + (ri + 8 * (mi & 1)) * 16;
#pragma unroll
    for (int s = 0; s < D / 32; ++s) {
      uint32_t a[4];
      ldmatrix_x4(a, row + (size_t)(2 * s) * (kBS * 16));
      mma_s8_16832(acc[m], a, qf[s][0], qf[s][1]);
    }
  }
}

// B-operand fragments of the GQA-packed query rows: row g of the N-tile is query
// head kvh*G + g; qf[s] = dims {32s+4t..+3} and {32s+16+4t..+3}.
template <int D>
__device__ __forceinline__ void load_q_frags(const int8_t* q, int b, int Hq, int kvh, int G, int lane,
                                             uint32_t (&qf)[D / 32][2]) {
  const int g = lane >> 2, t = lane & 3;
  const int8_t* row = q + ((size_t)b * Hq + kvh * G + g) * D;
#pragma unroll
  for (int s = 0; s < D / 32; ++s) {
    qf[s][0] = g < G ? __ldg(reinterpret_cast<const uint32_t*>(row + 32 * s + 4 * t)) : 0u;
    qf[s][1] = g < G ? __ldg(reinterpret_cast<const uint32_t*>(row + 32 * s + 16 + 4 * t)) : 0u;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) int8_decode_kernel(DecodeParams p, int nslots) {
  constexpr int NDT = D / 16 / kCWarps;  // PV head-dim tiles per warp
  constexpr int kPage = D * kBS;
  constexpr int kItem = kPart * D;
  extern __shared__ __align__(1024) uint8_t smem[];
  const SmemLayout lay = decode_layout(D, p.Hkv, nslots);
  int8_t* ring = reinterpret_cast<int8_t*>(smem + lay.ring);
  float* scales = reinterpret_cast<float*>(smem + lay.scales);
  float* wbuf = reinterpret_cast<float*>(smem + lay.wbuf);
  uint2* wqf = reinterpret_cast<uint2*>(smem + lay.wqf);
  float* swr = reinterpret_cast<float*>(smem + lay.swr);
  float* redmax = reinterpret_cast<float*>(smem + lay.redmax);
  float* redsum = reinterpret_cast<float*>(smem + lay.redsum);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint64_t* empty = full + nslots;
  int* ctrl = reinterpret_cast<int*>(smem + lay.ctrl);
  volatile int* abort_flag = ctrl + 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.B, Hkv = p.Hkv, G = p.G, Hq = p.Hq;
  const int N = gridDim.x, c = blockIdx.x;
  const int maxL = p.max_blocks * kBS;
  const int scale_floats = kPart * Hkv;  // one of sK / sV for one unit

  // ---- work split: every CTA scans seq_lens (warp 0) ----
  if (warp == 0) {
    long long total = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int u = 0;
      if (b < B) {
        const int raw = p.seq_lens[b];
        if (raw > maxL) record_error(2);
        const int L = clamp_len(raw, maxL);
        u = (L + kPart - 1) / kPart * Hkv;
        if (L == 0 && b % N == c) {  // empty sequence: zero rows
          float* o = p.out + (size_t)b * Hq * D;
          for (int i = 0; i < Hq * D; ++i) o[i] = 0.f;
        }
      }
      for (int o = 16; o >= 1; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
      total += u;
    }
    const long long U = total;
    // Only the first min(N, U) CTAs take units, so every working CTA has at
    // least one and the CTAs covering a pair are consecutive.
    const int Nw = (int)(U < N ? U : N);
    const long long ub = c < Nw ? U * c / Nw : 0, ue = c < Nw ? U * (c + 1) / Nw : 0;
    if (lane == 0) {
      ctrl[0] = (int)(ue - ub);
      ctrl[8] = 0;
      ctrl[10] = Nw;
    }
    if (ue > ub) {
      // find the sequence holding unit ub
      long long run = 0;
      for (int b0 = 0; b0 < B; b0 += 32) {
        const int b = b0 + lane;
        int u = 0;
        if (b < B) u = (clamp_len(p.seq_lens[b], maxL) + kPart - 1) / kPart * Hkv;
        int incl = u;
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const long long ex = run + incl - u, in = run + incl;
        const unsigned hit = __ballot_sync(0xffffffffu, u > 0 && ex <= ub && ub < in);
        if (hit) {
          const int src = __ffs(hit) - 1;
          if (lane == src) {
            const int L = clamp_len(p.seq_lens[b], maxL);
            const int np = (L + kPart - 1) / kPart;
            const long long local = ub - ex;
            ctrl[1] = b;
            ctrl[2] = (int)(local / np);
            ctrl[3] = (int)(local % np);
            ctrl[4] = (int)(ex & 0x7fffffff);
            ctrl[5] = (int)(ex >> 31);
          }
          break;
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        ctrl[6] = (int)(U & 0x7fffffff);
        ctrl[7] = (int)(U >> 31);
      }
    }
  }
  if (tid == 0) {
    for (int s = 0; s < nslots; ++s) {
      mbar_init(&full[s], 32);
      mbar_init(&empty[s], kCWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int n_units = ctrl[0];
  if (n_units <= 0) return;
  Walk w0;
  w0.b = ctrl[1];
  w0.kvh = ctrl[2];
  w0.part = ctrl[3];
  w0.ub = (long long)ctrl[4] | ((long long)ctrl[5] << 31);
  w0.L = clamp_len(p.seq_lens[w0.b], maxL);
  w0.np = (w0.L + kPart - 1) / kPart;
  const long long U = (long long)ctrl[6] | ((long long)ctrl[7] << 31);
  const int Nw = ctrl[10];

  if (warp == kCWarps) {
    // ================= producer warp =================
    const int8_t* kc = static_cast<const int8_t*>(p.k_cache);
    const int8_t* vc = static_cast<const int8_t*>(p.v_cache);
    const uint64_t pol = policy_evict_first();
    Walk wk = w0;
    const int j = lane & 15;
    for (int i = 0; i < n_units; ++i) {
      const int t0 = wk.part * kPart;
      const int nblk = min(kPart / kBS, (wk.L - t0 + kBS - 1) / kBS);
      int blk = -1;
      if (j < nblk) {
        blk = p.block_tables[(size_t)wk.b * p.max_blocks + wk.part * (kPart / kBS) + j];
        if (blk < 0 || blk >= p.num_blocks) {
          record_error(2);
          blk = -1;
        }
      }
      const bool page_ok = lane < 16 && blk >= 0;
      const bool scale_ok = lane >= 16 && blk >= 0;
      const uint32_t n_pages = __popc(__ballot_sync(0xffffffffu, page_ok));
      const uint32_t n_srows = __popc(__ballot_sync(0xffffffffu, scale_ok));
      const uint32_t srow_bytes = kBS * Hkv * sizeof(float);
      // K item (+ both scale rows)
      {
        const int item = 2 * i, slot = item % nslots;
        if (item >= nslots) pipe_wait(&empty[slot], ((item / nslots) - 1) & 1, abort_flag);
        if (lane == 0) mbar_expect_tx(&full[slot], n_pages * kPage + n_srows * 2 * srow_bytes);
        __syncwarp();
        if (page_ok)
          bulk_g2s_hint(ring + (size_t)slot * kItem + (size_t)j * kPage, kc + ((size_t)blk * Hkv + wk.kvh) * kPage,
                        kPage, &full[slot], pol);
        if (scale_ok) {
          float* ss = scales + (size_t)(i % lay.nsslots) * 2 * scale_floats;
          bulk_g2s_hint(ss + j * kBS * Hkv, p.k_scale + (size_t)blk * kBS * Hkv, srow_bytes, &full[slot], pol);
          bulk_g2s_hint(ss + scale_floats + j * kBS * Hkv, p.v_scale + (size_t)blk * kBS * Hkv, srow_bytes,
                        &full[slot], pol);
        }
        mbar_arrive(&full[slot]);
      }
      // V item
      {
        const int item = 2 * i + 1, slot = item % nslots;
        if (item >= nslots) pipe_wait(&empty[slot], ((item / nslots) - 1) & 1, abort_flag);
        if (lane == 0) mbar_expect_tx(&full[slot], n_pages * kPage);
        __syncwarp();
        if (page_ok)
          bulk_g2s_hint(ring + (size_t)slot * kItem + (size_t)j * kPage, vc + ((size_t)blk * Hkv + wk.kvh) * kPage,
                        kPage, &full[slot], pol);
        mbar_arrive(&full[slot]);
      }
      walk_next(wk, p.seq_lens, B, Hkv, maxL);
    }
    return;
  }

  // ================= consumer warps =================
  const int g = lane >> 2, t = lane & 3;
  const float c_scale = p.sm_scale;
  Walk wk = w0;
  int cur_pair = -1;
  uint32_t qf[D / 32][2];
  float sq[2] = {0.f, 0.f};
  float o[NDT][4];
  float Mrun[2], Lrun[2];
  for (int i = 0; i < n_units; ++i) {
    const int pair = wk.b * Hkv + wk.kvh;
    if (pair != cur_pair) {
      cur_pair = pair;
      load_q_frags<D>(static_cast<const int8_t*>(p.q), wk.b, Hq, wk.kvh, G, lane, qf);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = 2 * t + r;
        sq[r] = row < G ? p.q_scale[(size_t)wk.b * Hq + wk.kvh * G + row] : 0.f;
        Mrun[r] = -INFINITY;
        Lrun[r] = 0.f;
      }
#pragma unroll
      for (int dt = 0; dt < NDT; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[dt][e] = 0.f;
    }
    const int t0 = wk.part * kPart;
    const int ntok = min(kPart, wk.L - t0);
    const float* sks = scales + (size_t)(i % lay.nsslots) * 2 * scale_floats;
    const float* svs = sks + scale_floats;

    // ---- K item: QK, scores, partition max ----
    const int kitem = 2 * i, kslot = kitem % nslots;
    pipe_wait(&full[kslot], (kitem / nslots) & 1, abort_flag);
    int acc[2][4];
    if (warp * kGroup < ntok) {
      qk_warp<D>(ring + (size_t)kslot * kItem, warp, lane, qf, acc);
    } else {
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[m][e] = 0;
    }
    float s[2][4], sv[2][4];
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = warp * kGroup + 16 * m + g + 8 * (e >> 1);
        const bool valid = tok < ntok;
        float sc = -INFINITY, vsc = 0.f;
        if (valid) {
          const float sk = sks[tok * Hkv + wk.kvh];
          vsc = svs[tok * Hkv + wk.kvh];
          sc = __fmul_rn(__fmul_rn(__fmul_rn((float)acc[m][e], sq[e & 1]), sk), c_scale);
        }
        s[m][e] = sc;
        sv[m][e] = vsc;
        mx[e & 1] = fmaxf(mx[e & 1], sc);
      }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[kslot]);
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int off = 4; off <= 16; off <<= 1) mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], off));
    if (g == 0) {
      redmax[warp * kRows + 2 * t] = mx[0];
      redmax[warp * kRows + 2 * t + 1] = mx[1];
    }
    named_bar_sync(1, kCWarps * 32);

    // ---- partition softmax: m_g, l_g, P, W = P * sV ----
    float mg[2], lg[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float m_ = -INFINITY;
#pragma unroll
      for (int w2 = 0; w2 < kCWarps; ++w2) m_ = fmaxf(m_, redmax[w2 * kRows + 2 * t + r]);
      mg[r] = m_;
    }
    float ps[2][4];
    float sum[2] = {0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pe = (s[m][e] == -INFINITY) ? 0.f : expf(__fsub_rn(s[m][e], mg[e & 1]));
        ps[m][e] = pe;
        sum[e & 1] += pe;
      }
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int off = 4; off <= 16; off <<= 1) sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], off);
    if (g == 0) {
      redsum[warp * kRows + 2 * t] = sum[0];
      redsum[warp * kRows + 2 * t + 1] = sum[1];
    }
    named_bar_sync(1, kCWarps * 32);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float l_ = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kCWarps; ++w2) l_ += redsum[w2 * kRows + 2 * t + r];
      lg[r] = l_;
    }
    float* wb = wbuf + (size_t)warp * kRows * kWStride;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = 2 * t + (e & 1);
        const int tg = 16 * m + g + 8 * (e >> 1);
        const float P = __fdiv_rn(ps[m][e], lg[e & 1]);
        wb[row * kWStride + tg] = (ps[m][e] > 0.f) ? __fmul_rn(P, sv[m][e]) : 0.f;
      }
    __syncwarp();
    // ---- W quantization of this warp's group, row g ----
    {
      const float4 w0v = *reinterpret_cast<const float4*>(wb + g * kWStride + 4 * t);
      const float4 w1v = *reinterpret_cast<const float4*>(wb + g * kWStride + 16 + 4 * t);
      const float wv[8] = {w0v.x, w0v.y, w0v.z, w0v.w, w1v.x, w1v.y, w1v.z, w1v.w};
      float A = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) A = fmaxf(A, wv[e]);
      A = fmaxf(A, __shfl_xor_sync(0xffffffffu, A, 1));
      A = fmaxf(A, __shfl_xor_sync(0xffffffffu, A, 2));
      const float sW = __fdiv_rn(A, 127.0f);
      int qv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) qv[e] = (A > 0.f) ? min(127, max(-127, __float2int_rn(__fdiv_rn(wv[e], sW)))) : 0;
      wqf[warp * 32 + lane] = make_uint2(pack_s8x4(qv[0], qv[1], qv[2], qv[3]), pack_s8x4(qv[4], qv[5], qv[6], qv[7]));
      if (t == 0) swr[warp * kRows + g] = (A > 0.f) ? sW : 0.f;
    }
    // ---- running merge of this partition into the CTA's state ----
    float wg[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float Mn = fmaxf(Mrun[r], mg[r]);
      const float a = (Mrun[r] == -INFINITY) ? 0.f : expf(Mrun[r] - Mn);
      wg[r] = lg[r] * expf(mg[r] - Mn);
      Lrun[r] = Lrun[r] * a + wg[r];
      Mrun[r] = Mn;
#pragma unroll
      for (int dt = 0; dt < NDT; ++dt) {
        o[dt][r] *= a;
        o[dt][2 + r] *= a;
      }
    }
    named_bar_sync(1, kCWarps * 32);

    // ---- V item: INT8 PV per group, rescaled by sW * merge weight ----
    const int vitem = 2 * i + 1, vslot = vitem % nslots;
    pipe_wait(&full[vslot], (vitem / nslots) & 1, abort_flag);
    {
      const int ngroups = (ntok + kGroup - 1) / kGroup;
      const int8_t* vpages = ring + (size_t)vslot * kItem;
      const int mi = lane >> 3, ri = lane & 7;
      for (int jg = 0; jg < ngroups; ++jg) {
        const uint2 bq = wqf[jg * 32 + lane];
        const float sc0 = swr[jg * kRows + 2 * t] * wg[0];
        const float sc1 = swr[jg * kRows + 2 * t + 1] * wg[1];
        const int8_t* vrow = vpages + (size_t)(2 * jg + (mi >> 1)) * kPage + (ri + 8 * (mi & 1)) * 16;
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt) {
          const int dtile = warp * NDT + dt;
          uint32_t a[4];
          ldmatrix_x4(a, vrow + dtile * 16 * 16);
          int pv[4] = {0, 0, 0, 0};
          mma_s8_16832(pv, a, bq.x, bq.y);
          o[dt][0] += (float)pv[0] * sc0;
          o[dt][1] += (float)pv[1] * sc1;
          o[dt][2] += (float)pv[2] * sc0;
          o[dt][3] += (float)pv[3] * sc1;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[vslot]);

    // ---- end of this CTA's segment of the (sequence, KV head) pair? ----
    Walk nx = wk;
    walk_next(nx, p.seq_lens, B, Hkv, maxL);
    const bool seg_end = (i == n_units - 1) || (nx.b * Hkv + nx.kvh != pair);
    if (seg_end) {
      const long long Up = wk.ub + (long long)wk.kvh * wk.np;
      const int cf = cta_of(Up, U, Nw), cl = cta_of(Up + wk.np - 1, U, Nw);
      if (cf == cl) {
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = 2 * t + (e & 1);
            const int d = (warp * NDT + dt) * 16 + g + 8 * (e >> 1);
            if (row < G) p.out[((size_t)wk.b * Hq + wk.kvh * G + row) * D + d] = o[dt][e] / Lrun[e & 1];
          }
      } else {
        float* part = p.ws_part + (size_t)(pair + c) * kSlotFloats(D);
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = 2 * t + (e & 1);
            const int d = (warp * NDT + dt) * 16 + g + 8 * (e >> 1);
            part[row * D + d] = o[dt][e];
          }
        if (warp == 0 && g == 0) {
          part[kRows * D + 2 * t] = Mrun[0];
          part[kRows * D + 2 * t + 1] = Mrun[1];
          part[kRows * D + kRows + 2 * t] = Lrun[0];
          part[kRows * D + kRows + 2 * t + 1] = Lrun[1];
        }
        __threadfence();
        named_bar_sync(1, kCWarps * 32);
        if (tid == 0) {
          const int old = atomicAdd(&p.ws_count[pair], 1);
          ctrl[9] = (old == cl - cf) ? 1 : 0;
        }
        named_bar_sync(1, kCWarps * 32);
        if (ctrl[9]) {
          __threadfence();
          for (int idx = tid; idx < G * D; idx += kCWarps * 32) {
            const int row = idx / D, d = idx % D;
            float M = -INFINITY;
            for (int cc = cf; cc <= cl; ++cc)
              M = fmaxf(M, __ldcg(p.ws_part + (size_t)(pair + cc) * kSlotFloats(D) + kRows * D + row));
            float num = 0.f, den = 0.f;
            for (int cc = cf; cc <= cl; ++cc) {
              const float* ps2 = p.ws_part + (size_t)(pair + cc) * kSlotFloats(D);
              const float e = expf(__ldcg(ps2 + kRows * D + row) - M);
              num += e * __ldcg(ps2 + row * D + d);
              den += e * __ldcg(ps2 + kRows * D + kRows + row);
            }
            p.out[((size_t)wk.b * Hq + wk.kvh * G + row) * D + d] = num / den;
          }
          if (tid == 0) p.ws_count[pair] = 0;
        }
      }
    }
    wk = nx;
  }
}

// Debug QK: one CTA per (sequence, KV head, 256-token partition); K pages are
// staged with plain 16-byte loads and the decode kernel's qk_warp computes the
// int32 accumulators.
template <int D>
__global__ void __launch_bounds__(256) debug_qk_kernel(DebugQKParams p) {
  constexpr int kPage = D * kBS;
  extern __shared__ __align__(1024) uint8_t smem[];
  int8_t* kp = reinterpret_cast<int8_t*>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nparts = (p.max_len + kPart - 1) / kPart;
  const int part = blockIdx.x % nparts;
  const int kvh = (blockIdx.x / nparts) % p.Hkv;
  const int b = blockIdx.x / nparts / p.Hkv;
  const int L = clamp_len(p.seq_lens[b], p.max_blocks * kBS);
  const int t0 = part * kPart;
  for (int i = tid; i < kPart / kBS * kPage / 16; i += blockDim.x) {
    const int jb = i / (kPage / 16), w16 = i % (kPage / 16);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (t0 + jb * kBS < L) {
      const int blk = p.block_tables[(size_t)b * p.max_blocks + part * (kPart / kBS) + jb];
      if (blk >= 0 && blk < p.num_blocks)
        val = __ldg(reinterpret_cast<const uint4*>(p.k_cache + ((size_t)blk * p.Hkv + kvh) * kPage) + w16);
      else
        record_error(2);
    }
    reinterpret_cast<uint4*>(kp)[i] = val;
  }
  __syncthreads();
  uint32_t qf[D / 32][2];
  load_q_frags<D>(p.q, b, p.Hq, kvh, p.G, lane, qf);
  int acc[2][4];
  qk_warp<D>(kp, warp, lane, qf, acc);
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int tok = t0 + warp * kGroup + 16 * m + g + 8 * (e >> 1);
      const int row = 2 * t + (e & 1);
      if (row < p.G && tok < p.max_len)
        p.acc[((size_t)b * p.Hq + kvh * p.G + row) * p.max_len + tok] = tok < L ? acc[m][e] : 0;
    }
}

int g_num_sms[64] = {0};

int num_sms(int device) {
  if (device < 0 || device >= 64) return 148;
  if (g_num_sms[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0) n = 148;
    g_num_sms[device] = n;
  }
  return g_num_sms[device];
}

int g_max_smem[64] = {0};

int max_smem_optin(int device) {
  if (device < 0 || device >= 64) return 227 * 1024;
  if (g_max_smem[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess || n <= 0)
      n = 227 * 1024;
    g_max_smem[device] = n;
  }
  return g_max_smem[device];
}

// Deepest ring that fits.
int pick_slots(int D, int Hkv, int smem_limit) {
  for (int ns = 8; ns >= 2; --ns)
    if (decode_layout(D, Hkv, ns).total <= (size_t)smem_limit) return ns;
  return 0;
}

template <int D>
cudaError_t launch_decode_d(const DecodeParams& p, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  const int ns = pick_slots(D, p.Hkv, max_smem_optin(dev));
  if (ns == 0) return cudaErrorInvalidConfiguration;
  const size_t smem = decode_layout(D, p.Hkv, ns).total;
  // Raise the dynamic shared-memory limit once per device (to the opt-in
  // maximum), so that launches captured into a CUDA graph make no attribute call.
  static int attr_set[64] = {0};
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(int8_decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         max_smem_optin(dev));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = 1;
  }
  int8_decode_kernel<D><<<p.grid, kThreads, smem, stream>>>(p, ns);
  return cudaGetLastError();
}

}  // namespace

int decode_grid(int device, int B, int Hkv, int max_blocks) {
  const long long max_units = (long long)B * Hkv * (((long long)max_blocks * kBS + kPart - 1) / kPart);
  long long g = num_sms(device);
  if (max_units < g) g = max_units;
  return (int)(g < 1 ? 1 : g);
}

size_t decode_workspace_bytes(int B, int Hkv, int D, int grid) {
  const size_t slots = (size_t)B * Hkv + (size_t)grid;
  size_t bytes = slots * kSlotFloats(D) * sizeof(float) + (size_t)B * Hkv * sizeof(int);
  return (bytes + 255) / 256 * 256;
}

I8KV_DEFINE_ERROR_ACCESSOR(read_error_decode)

cudaError_t launch_int8_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.D == 256) return launch_decode_d<256>(p, stream);
  return launch_decode_d<128>(p, stream);
}

cudaError_t launch_debug_qk(const DebugQKParams& p, cudaStream_t stream) {
  const int nparts = (p.max_len + kPart - 1) / kPart;
  const long long grid = (long long)p.B * p.Hkv * nparts;
  if (grid == 0) return cudaSuccess;
  const size_t smem = (size_t)kPart * p.D;
  cudaError_t e;
  if (p.D == 256) {
    e = cudaFuncSetAttribute(debug_qk_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    debug_qk_kernel<256><<<(unsigned)grid, 256, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(debug_qk_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    debug_qk_kernel<128><<<(unsigned)grid, 256, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace i8kv
