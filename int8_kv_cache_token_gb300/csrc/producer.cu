// producer.cu -- the fused KV producer: per-(token, head) absmax INT8
// quantization of K, V (and optionally Q) and the scatter into the paged cache.
//
// Source: "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化", §2.1 (the
// quantization rule), §2.2 (the fused producer: absmax, scale, quantize, paged
// write and scale write in one kernel, query quantized once) and §2.3 (layouts).
//
// GB300 shape: a persistent, warp-specialized CTA per SM, fed by bulk copies.
//  * Work unit = 16 consecutive tokens (one cache block's worth) x a group of
//    heads of one tensor: per tile of 16 tokens the V units, then the K units,
//    then the Q units, each holding up to 1024 / D heads (token rows of at most
//    2 KB).  CTA c takes the contiguous unit range [c U / N, (c+1) U / N).
//  * Loader warp: per unit, one bulk copy per token row (16 rows, each the
//    unit's heads of one token, contiguous in the [T, H, D] input) into a ring
//    slot; rows sit 16 bytes apart more than their length so the compute warps'
//    16-byte reads of the same run in consecutive tokens fall on different
//    banks.  Per tile it also publishes the tile's slots, positions and the
//    "one whole cache block in order" flag (and, fused, bulk-copies the tile's
//    cos/sin table rows) into a ring of tile entries.
//  * 15 compute warps: the unit's heads are its tasks, handed out round-robin
//    (the CTA's task t goes to warp t % 15, so about two units are in work at
//    once); a task is one head over the tile's 16 tokens.  With the loader the
//    CTA has 16 warps, four per SM sub-partition, at 128 registers each.
//    A vector (token, head) is held by D/32 lanes, 32 elements per lane in two
//    16-element runs, so a warp pass covers VPW = 1024 / D tokens.  Lane =
//    c * VPW + token, with c the lane's place in its vector: the 8 lanes of a
//    quarter-warp then read the same run of 8 consecutive token rows, which the
//    16-byte row padding puts on 8 different bank groups.  The absmax is a max
//    over the lane's 32 values, then xor-shuffles across the vector's lanes
//    (distances VPW, 2 VPW, ...).
//  * Outputs leave as 16-byte stores: K and Q codes per run (K's 16-dim chunk
//    layout makes a run contiguous), V per warp: when the tile fills one whole
//    block in order (the common prefill case) the task's 16 x D codes are
//    staged in the slot itself, over the head's bf16 rows that only this warp
//    reads, and written transposed (token-inner), 16 bytes per (dim) row;
//    otherwise each lane writes its codes byte by byte.
//
// Bit-exactness: scale = amax / 127 and x / scale are IEEE fp32 divisions,
// codes are round-half-to-even; the build does not use fast-math.
//
// The fused variant ([KV] §2.2 step 2, §5.3) first applies a per-head RMSNorm
// and rotate-half RoPE to each Q and K vector in fp32, every operation a single
// correctly rounded one in a fixed order, so its cache bytes are reproducible
// too.  The lane's two runs are chosen so that RoPE never leaves the lane: with
// hr = rotary_dim / 32 rotary runs per half, lane c < hr holds runs c and
// c + hr (dims i and i + rotary_dim/2 together), the other lanes hold two
// consecutive runs of the unrotated tail.  The RMSNorm sum keeps its balanced
// tree in index order: each run's 16 squares are summed as a tree in the lane,
// the run sums meet in a small per-warp shared buffer, and every lane of the
// vector sums them as the same tree over runs.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace i8kv {

namespace {

constexpr int kTok = 16;          // tokens per tile (the cache block size)
constexpr int kNCW = 15;          // compute warps
constexpr int kProdThreads = (kNCW + 1) * 32;
constexpr int kTR = 3;            // tile entries in flight
constexpr int kMaxSlots = 8;
constexpr int kMaxSmem = 232448;  // 227 KB of dynamic shared memory per CTA

struct TileMeta {
  int slot[kTok];  // cache slot; -1: no K/V write
  int pos[kTok];   // table row (fused with rotation), else 0; -1: no such token or token skipped
  int aligned;     // the 16 tokens fill one cache block in order
  int pad[3];
};

// Geometry of one call (host-computed).
struct ProdGeo {
  long long units;  // work units of the call
  int upt;          // units per tile: nkv V units, nkv K units, nq Q units
  int kvh, qh;      // heads per K/V unit, per Q unit
  int nkv, nq;
  int S;            // ring slots
  int row_stride;   // bytes between token rows in a slot
  int slot_bytes;
  int off_nscr, off_meta, off_cs, off_sm, off_w, off_bar;
  int smem;
};

// mbarrier arrival counting `count` arrivals at once.
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t count) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(count)
      : "memory");
}

// Bounded wait that also gives up when another role of the CTA aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      record_error(1);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// 16 bf16 (two 16-byte words) to fp32.
__device__ __forceinline__ void bf16x16_to_f32(uint4 a, uint4 b, float* x) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 pack_codes16(const uint32_t* q) {
  uint32_t pk[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    pk[j] = __byte_perm(__byte_perm(q[4 * j], q[4 * j + 1], 0x0040), __byte_perm(q[4 * j + 2], q[4 * j + 3], 0x0040),
                        0x5410);
  return make_uint4(pk[0], pk[1], pk[2], pk[3]);
}

// Quantize the vector whose 32 elements this lane holds (the lanes VPW apart
// hold one vector).  Every lane of the warp calls this (the absmax shuffles
// across the whole warp).  Returns the vector's scale; codes of the lane's two
// runs in ca, cb.
//  Codes: round half to even by adding 1.5 * 2^23 (the fp32 sum keeps the
//  integer part of x / scale in its low mantissa bits, so its low byte is the
//  two's-complement code).  |x / scale| <= amax / RN(amax / 127) < 127.5, so no
//  code ever needs clamping to [-127, 127].
template <int VPW>
__device__ __forceinline__ float quantize32(const float (&x)[32], uint4& ca, uint4& cb) {
  float m0 = 0.f, m1 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    m0 = fmaxf(m0, fabsf(x[2 * i]));
    m1 = fmaxf(m1, fabsf(x[2 * i + 1]));
  }
  float amax = fmaxf(m0, m1);
#pragma unroll
  for (int o = 16; o >= VPW; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = div127(amax);  // amax / 127, correctly rounded
  uint32_t q[32];
  if (amax > 0.f) {
    div_rne_row(x, scale, __frcp_rn(scale), q);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) q[i] = 0;
  }
  ca = pack_codes16(q);
  cb = pack_codes16(q + 16);
  return amax > 0.f ? scale : 0.f;
}

__device__ __forceinline__ void store_bf16x16(uint16_t* dst, const float* x) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = bf16x2_rn(x[2 * i], x[2 * i + 1]);
  *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(dst + 8) = make_uint4(w[4], w[5], w[6], w[7]);
}

// Sum of the squares of 16 values as a balanced tree in index order.
__device__ __forceinline__ float sum_sq16(const float* x) {
  float s[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float lo, hi;
    const uint64_t v = f2(x[2 * i], x[2 * i + 1]);
    f2_split(mul2(v, v), lo, hi);
    s[i] = __fadd_rn(lo, hi);
  }
#pragma unroll
  for (int n = 4; n >= 1; n >>= 1)
#pragma unroll
    for (int i = 0; i < n; ++i) s[i] = __fadd_rn(s[2 * i], s[2 * i + 1]);
  return s[0];
}

// x[i] *= m[i] for the lane's 16 values of one run (each product rounded once).
__device__ __forceinline__ void mul16(float* x, const float* m) {
#pragma unroll
  for (int j4 = 0; j4 < 4; ++j4) {
    const float4 f = *reinterpret_cast<const float4*>(m + 4 * j4);
    f2_split(mul2(f2(x[4 * j4], x[4 * j4 + 1]), f2(f.x, f.y)), x[4 * j4], x[4 * j4 + 1]);
    f2_split(mul2(f2(x[4 * j4 + 2], x[4 * j4 + 3]), f2(f.z, f.w)), x[4 * j4 + 2], x[4 * j4 + 3]);
  }
}

// 128 registers: four warps of 32 threads per SM sub-partition fill its 16 K.
template <int D, bool kFused>
__global__ void __launch_bounds__(kProdThreads, 1) kv_quant_write_kernel(ProducerParams p, ProdGeo g) {
  constexpr int LPV = D / 32;    // lanes per vector
  constexpr int VPW = 32 / LPV;  // vectors (tokens) per warp pass
  constexpr int R = D / 16;      // 16-element runs per vector
  extern __shared__ __align__(1024) uint8_t dsm[];
  uint8_t* ring = dsm;
  TileMeta* meta = reinterpret_cast<TileMeta*>(dsm + g.off_meta);
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm + g.off_bar);
  uint64_t* freeb = full + kMaxSlots;
  uint64_t* meta_full = freeb + kMaxSlots;
  uint64_t* tile_free = meta_full + kTR;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tile_free + kTR);
  // slot_use[s]: the use of slot s whose copies the loader has issued.  A
  // compute warp waits only on the slots of the units it has a task in, so it
  // may reach use u of a slot before use u - 1 has landed; the full barrier's
  // parity test alone would then take the older phase for this one.  Waiting
  // for the stamp first keeps every waiter within one phase of the barrier.
  volatile int* slot_use = abort_flag + 4;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rd = kFused ? p.rd : 0;
  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < g.S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&freeb[i], kNCW);
      slot_use[i] = -1;
    }
    for (int i = 0; i < kTR; ++i) {
      mbar_init(&meta_full[i], 1);
      mbar_init(&tile_free[i], kNCW);
    }
    fence_mbar_init();
  }
  // From here on the kernel reads what earlier work on the stream writes.
  griddep_wait();
  griddep_launch_dependents();
  if constexpr (kFused) {
    float* s_w = reinterpret_cast<float*>(dsm + g.off_w);
    for (int i = tid; i < 2 * D; i += blockDim.x) {
      const uint16_t* w = i < D ? p.q_norm_w : p.k_norm_w;
      s_w[i] = w ? bf16_bits_to_float(__ldg(w + i % D)) : 0.f;
    }
    if (p.k_smooth) {
      float* s_sm = reinterpret_cast<float*>(dsm + g.off_sm);  // s [Hkv][D], then RN(1/s) [Hkv][D]
      for (int i = tid; i < p.Hkv * D; i += blockDim.x) {
        const float f = __ldg(p.k_smooth + i);
        s_sm[i] = f;
        s_sm[p.Hkv * D + i] = __frcp_rn(f);
      }
    }
  }
  __syncthreads();

  const long long u0 = (long long)blockIdx.x * g.units / gridDim.x;
  const long long u1 = (long long)(blockIdx.x + 1) * g.units / gridDim.x;
  const int T = p.T;
  const long long pool_slots = (long long)p.num_blocks * kTok;

  if (warp == kNCW) {
    // ------------------------------------------------------------ loader warp
    const uint64_t l2_first = policy_evict_first();
    // Tile metadata is read one tile ahead (registers), published just before
    // the loader could block on a slot that this tile's units may occupy.
    auto read_meta = [&](long long n, int& s, int& pos) {
      s = -1;
      pos = -1;
      const long long t = n * kTok + lane;
      if (lane < kTok && t < T) {
        s = __ldg(p.slots + t);
        pos = (kFused && rd > 0) ? __ldg(p.positions + t) : 0;
      }
    };
    long long cur = -1;
    int tl = -1;
    bool pending = false;
    int m_s = -1, m_pos = -1, nx_s = -1, nx_pos = -1;
    read_meta(u0 / g.upt, nx_s, nx_pos);
    auto publish = [&]() -> bool {
      pending = false;
      const int te = tl % kTR;
      if (tl >= kTR && !wait_or_abort(&tile_free[te], ((tl / kTR) - 1) & 1, abort_flag)) return false;
      const bool present = lane < kTok && cur * kTok + lane < T;
      int s = present ? m_s : -1, pos = present ? m_pos : -1;
      if (s >= pool_slots) {
        record_error(2);
        s = -1;
      }
      if (kFused && rd > 0 && present && (pos < 0 || pos >= p.max_pos)) {  // outside the table: skipped
        record_error(4);
        pos = -1;
        s = -1;
      }
      TileMeta* m = meta + te;
      if (lane < kTok) {
        m->slot[lane] = s;
        m->pos[lane] = pos;
      }
      const int s0 = __shfl_sync(0xffffffffu, s, 0);
      const bool al = __all_sync(0xffffffffu, lane >= kTok || (s0 >= 0 && s0 % kTok == 0 && s == s0 + lane));
      if (lane == 0) m->aligned = al ? 1 : 0;
      __syncwarp();
      const bool cp = kFused && rd > 0 && lane < kTok && pos >= 0;
      const uint32_t n_cp = __popc(__ballot_sync(0xffffffffu, cp));
      if (lane == 0) {
        if (n_cp) mbar_expect_tx(&meta_full[te], n_cp * rd * 4);
        mbar_arrive(&meta_full[te]);
      }
      if (cp) {
        float* cs = reinterpret_cast<float*>(dsm + g.off_cs) + ((size_t)te * kTok + lane) * (rd + 4);
        bulk_g2s(cs, p.cos_sin + (size_t)pos * rd, rd * 4, &meta_full[te]);
      }
      return true;
    };
    // The unit's tile n, its place k in the tile, its slot s and the slot's use
    // advance by increments (no divisions per unit).
    const int nloc = (int)(u1 - u0);
    long long n = u0 / g.upt;
    int k = (int)(u0 - n * g.upt), s = 0, use = 0, i = 0;
    bool ok = true;
    for (; i < nloc; ++i) {
      if (i == 0 || k == 0) {
        if (pending && !publish()) {
          ok = false;
          break;
        }
        cur = n;
        ++tl;
        m_s = nx_s;
        m_pos = nx_pos;
        read_meta(n + 1, nx_s, nx_pos);
        pending = true;
      }
      if (use > 0) {
        if (pending && !publish()) {
          ok = false;
          break;
        }
        if (!wait_or_abort(&freeb[s], (uint32_t)((use - 1) & 1), abort_flag)) {
          ok = false;
          break;
        }
      }
      const int kind = k < g.nkv ? 1 : (k < 2 * g.nkv ? 0 : 2);  // 0 K, 1 V, 2 Q
      const int nh = kind == 2 ? g.qh : g.kvh;
      const int h0 = (kind == 2 ? k - 2 * g.nkv : (kind == 1 ? k : k - g.nkv)) * nh;
      const int H = kind == 2 ? p.Hq : p.Hkv;
      const uint16_t* src = kind == 0 ? p.k : (kind == 1 ? p.v : p.q);
      const int ntv = (int)min((long long)kTok, (long long)T - n * kTok);
      const uint32_t rb = (uint32_t)nh * D * 2;
      if (lane == 0) {
        slot_use[s] = use;
        mbar_expect_tx(&full[s], ntv * rb);
        mbar_arrive(&full[s]);
      }
      if (lane < ntv)  // the bf16 rows are read once: L2 lets them go first
        bulk_g2s_hint(ring + (size_t)s * g.slot_bytes + (size_t)lane * g.row_stride,
                      src + ((size_t)(n * kTok + lane) * H + h0) * D, rb, &full[s], l2_first);
      if (++s == g.S) {
        s = 0;
        ++use;
      }
      if (++k == g.upt) {
        k = 0;
        ++n;
      }
    }
    if (ok && pending) ok = publish();
    if (!ok) {
      // Aborted: hold the CTA (and its shared memory) until every copy issued
      // into it has landed.  Slot s's last issued item is the newest local
      // unit j < i with j % S == s.
      *abort_flag = 1;
      for (int sl = 0; sl < g.S; ++sl) {
        const int last = i - 1 - ((i - 1 - sl) % g.S + g.S) % g.S;
        if (last < 0 || last >= i) continue;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&full[sl], (uint32_t)((last / g.S) & 1)) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    return;
  }

  // --------------------------------------------------------------- compute warps
  const int c = lane / VPW, vi = lane % VPW;  // place in the vector, token of the pass
  const int hr = rd / 32;  // rotary runs per half
  const int ra = c < hr ? c : 2 * hr + 2 * (c - hr);
  const int rb = c < hr ? c + hr : ra + 1;
  const bool k_copy = kFused && p.k_out != nullptr;
  const float* s_w = reinterpret_cast<const float*>(dsm + g.off_w);
  const float* s_sm = reinterpret_cast<const float*>(dsm + g.off_sm);
  constexpr int NS = R + 4;  // run sums per vector, padded (bank spread)
  float* nscr = reinterpret_cast<float*>(dsm + g.off_nscr) + warp * VPW * NS;
  const int G = p.q ? p.Hq / p.Hkv : 1;

  // Per unit: its tile n and place k, its slot s and the slot's use, and the
  // CTA's task count modulo kNCW, all advanced by increments.
  const int nloc = (int)(u1 - u0);
  long long n = u0 / g.upt;
  int k = (int)(u0 - n * g.upt), s = 0, use = 0, tmod = 0, tl = -1;
  auto advance = [&](int nh) {
    tmod += nh;
    if (tmod >= kNCW) tmod -= kNCW;
    if (++s == g.S) {
      s = 0;
      ++use;
    }
    if (++k == g.upt) {
      k = 0;
      ++n;
    }
  };
  for (int i = 0; i < nloc; ++i) {
    if (i == 0 || k == 0) {
      if (tl >= 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&tile_free[tl % kTR]);
      }
      ++tl;
      if (!wait_or_abort(&meta_full[tl % kTR], (uint32_t)((tl / kTR) & 1), abort_flag)) break;
    }
    const int kind = k < g.nkv ? 1 : (k < 2 * g.nkv ? 0 : 2);
    const int nh = kind == 2 ? g.qh : g.kvh;
    int hp = warp - tmod;  // this warp's task in the unit
    if (hp < 0) hp += kNCW;
    if (hp >= nh) {
      advance(nh);
      continue;
    }
    if (slot_use[s] != use) {
      const uint64_t t0 = global_timer_ns();
      while (slot_use[s] != use && !*abort_flag) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          record_error(1);
          *abort_flag = 1;
        }
      }
      if (*abort_flag) break;
    }
    if (!wait_or_abort(&full[s], (uint32_t)(use & 1), abort_flag)) break;

    const TileMeta* m = meta + tl % kTR;
    const int h = (kind == 2 ? k - 2 * g.nkv : (kind == 1 ? k : k - g.nkv)) * nh + hp;
    const int H = kind == 2 ? p.Hq : p.Hkv;
    uint8_t* base = ring + (size_t)s * g.slot_bytes + (size_t)hp * D * 2;
    const bool v_block = kind == 1 && m->aligned;
    const bool norm = kFused && ((kind == 0 && p.k_norm_w) || (kind == 2 && p.q_norm_w));
#pragma unroll 1
    for (int ps = 0; ps < kTok / VPW; ++ps) {
      const int tok = ps * VPW + vi;
      const int slot = m->slot[tok];
      bool act = m->pos[tok] >= 0;
      if (kind == 1) act = act && slot >= 0;
      if (kind == 0) act = act && (slot >= 0 || k_copy);
      const long long t = n * kTok + tok;
      const uint8_t* row = base + (size_t)tok * g.row_stride;
      float x[32];
      bf16x16_to_f32(*reinterpret_cast<const uint4*>(row + 32 * ra), *reinterpret_cast<const uint4*>(row + 32 * ra + 16),
                     x);
      bf16x16_to_f32(*reinterpret_cast<const uint4*>(row + 32 * rb), *reinterpret_cast<const uint4*>(row + 32 * rb + 16),
                     x + 16);
      if constexpr (kFused) {
        if (kind != 1) {
          if (norm) {
            nscr[vi * NS + ra] = sum_sq16(x);
            nscr[vi * NS + rb] = sum_sq16(x + 16);
            __syncwarp();
            float rs[R];
#pragma unroll
            for (int j = 0; j < R / 4; ++j) {
              const float4 f = *reinterpret_cast<const float4*>(nscr + vi * NS + 4 * j);
              rs[4 * j] = f.x;
              rs[4 * j + 1] = f.y;
              rs[4 * j + 2] = f.z;
              rs[4 * j + 3] = f.w;
            }
            __syncwarp();
#pragma unroll
            for (int w2 = R / 2; w2 >= 1; w2 >>= 1)
#pragma unroll
              for (int j = 0; j < w2; ++j) rs[j] = __fadd_rn(rs[2 * j], rs[2 * j + 1]);
            const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(rs[0], 1.0f / D), p.eps)));
            const uint64_t inv2 = f2(inv, inv);
            const float* w = s_w + (kind == 0 ? D : 0);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const float* wr = w + 16 * (half ? rb : ra);
              float* xr = x + 16 * half;
#pragma unroll
              for (int j4 = 0; j4 < 4; ++j4) {
                const float4 f = *reinterpret_cast<const float4*>(wr + 4 * j4);
                f2_split(mul2(mul2(f2(xr[4 * j4], xr[4 * j4 + 1]), inv2), f2(f.x, f.y)), xr[4 * j4], xr[4 * j4 + 1]);
                f2_split(mul2(mul2(f2(xr[4 * j4 + 2], xr[4 * j4 + 3]), inv2), f2(f.z, f.w)), xr[4 * j4 + 2],
                         xr[4 * j4 + 3]);
              }
            }
          }
          if (c < hr) {
            // rotate-half: a = x_i (run ra), b = x_{i + rd/2} (run rb = ra + hr).
            // Products rounded, then a scalar add / subtract (no contraction).
            // table rows sit rd + 4 floats apart (bank spread)
            const float* cs =
                reinterpret_cast<const float*>(dsm + g.off_cs) + ((size_t)(tl % kTR) * kTok + tok) * (rd + 4);
            const float* cr = cs + 16 * ra;
            const float* sr = cs + rd / 2 + 16 * ra;
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              const float4 cv = *reinterpret_cast<const float4*>(cr + 4 * j4);
              const float4 sv = *reinterpret_cast<const float4*>(sr + 4 * j4);
              float ac[4], bs[4], bc[4], as[4];
              f2_split(mul2(f2(x[4 * j4], x[4 * j4 + 1]), f2(cv.x, cv.y)), ac[0], ac[1]);
              f2_split(mul2(f2(x[4 * j4 + 2], x[4 * j4 + 3]), f2(cv.z, cv.w)), ac[2], ac[3]);
              f2_split(mul2(f2(x[16 + 4 * j4], x[16 + 4 * j4 + 1]), f2(sv.x, sv.y)), bs[0], bs[1]);
              f2_split(mul2(f2(x[16 + 4 * j4 + 2], x[16 + 4 * j4 + 3]), f2(sv.z, sv.w)), bs[2], bs[3]);
              f2_split(mul2(f2(x[16 + 4 * j4], x[16 + 4 * j4 + 1]), f2(cv.x, cv.y)), bc[0], bc[1]);
              f2_split(mul2(f2(x[16 + 4 * j4 + 2], x[16 + 4 * j4 + 3]), f2(cv.z, cv.w)), bc[2], bc[3]);
              f2_split(mul2(f2(x[4 * j4], x[4 * j4 + 1]), f2(sv.x, sv.y)), as[0], as[1]);
              f2_split(mul2(f2(x[4 * j4 + 2], x[4 * j4 + 3]), f2(sv.z, sv.w)), as[2], as[3]);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                x[4 * j4 + e] = __fsub_rn(ac[e], bs[e]);
                x[16 + 4 * j4 + e] = __fadd_rn(bc[e], as[e]);
              }
            }
          }
          if (act) {
            uint16_t* cpy = kind == 0 ? p.k_out : p.q_out;
            if (cpy) {
              uint16_t* dst = cpy + ((size_t)t * H + h) * D;
              store_bf16x16(dst + 16 * ra, x);
              store_bf16x16(dst + 16 * rb, x + 16);
            }
          }
          if (p.k_smooth) {
            // K: times RN(1/s[h]); Q: times s[h / G]
            const float* f = kind == 0 ? s_sm + (size_t)p.Hkv * D + (size_t)h * D : s_sm + (size_t)(h / G) * D;
            mul16(x, f + 16 * ra);
            mul16(x + 16, f + 16 * rb);
          }
        }
      }
      uint4 ca, cb;
      const float scale = quantize32<VPW>(x, ca, cb);
      if (v_block) {
        // codes over the head's own bf16 rows, once every lane has read its values
        __syncwarp();
        uint8_t* crow = base + (size_t)tok * g.row_stride;
        *reinterpret_cast<uint4*>(crow + 16 * ra) = ca;
        *reinterpret_cast<uint4*>(crow + 16 * rb) = cb;
      }
      if (!act) continue;
      if (kind == 2) {
        if (kFused && !p.q_i8) continue;
        int8_t* dst = p.q_i8 + ((size_t)t * p.Hq + h) * D;
        *reinterpret_cast<uint4*>(dst + 16 * ra) = ca;
        *reinterpret_cast<uint4*>(dst + 16 * rb) = cb;
        if (c == 0) p.q_scale[(size_t)t * p.Hq + h] = scale;
        continue;
      }
      if (slot < 0) continue;  // K copied to k_out only
      const int blk = slot / kTok, off = slot % kTok;
      const size_t sidx = (size_t)slot * p.Hkv + h;
      if (kind == 0) {
        int8_t* dst = p.k_cache + (((size_t)blk * p.Hkv + h) * R * kTok + off) * 16;
        *reinterpret_cast<uint4*>(dst + (size_t)ra * kTok * 16) = ca;
        *reinterpret_cast<uint4*>(dst + (size_t)rb * kTok * 16) = cb;
        if (c == 0) p.k_scale[sidx] = scale;
      } else {
        if (!v_block) {
          int8_t* dst = p.v_cache + ((size_t)blk * p.Hkv + h) * D * kTok + off;
          const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w}, wb[4] = {cb.x, cb.y, cb.z, cb.w};
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            dst[(size_t)(16 * ra + e) * kTok] = (int8_t)((wa[e >> 2] >> (8 * (e & 3))) & 0xff);
            dst[(size_t)(16 * rb + e) * kTok] = (int8_t)((wb[e >> 2] >> (8 * (e & 3))) & 0xff);
          }
        }
        if (c == 0) p.v_scale[sidx] = scale;
      }
    }
    if (v_block) {
      // The task's 16 x D codes, written token-inner: lane d4 reads 4 dims of
      // the 16 token rows (4 bytes each), transposes the 4x4 byte tiles with
      // byte permutes and writes one 16-byte row per dim.
      __syncwarp();
      int8_t* dst = p.v_cache + ((size_t)(m->slot[0] / kTok) * p.Hkv + h) * D * kTok;
#pragma unroll
      for (int d4 = lane; d4 < D / 4; d4 += 32) {
        uint32_t o[4][4];  // [dim j][token group]
#pragma unroll
        for (int tg = 0; tg < 4; ++tg) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) w[e] = *reinterpret_cast<const uint32_t*>(base + (size_t)(4 * tg + e) * g.row_stride + 4 * d4);
          const uint32_t x0 = __byte_perm(w[0], w[1], 0x5140), x1 = __byte_perm(w[0], w[1], 0x7362);
          const uint32_t y0 = __byte_perm(w[2], w[3], 0x5140), y1 = __byte_perm(w[2], w[3], 0x7362);
          o[0][tg] = __byte_perm(x0, y0, 0x5410);
          o[1][tg] = __byte_perm(x0, y0, 0x7632);
          o[2][tg] = __byte_perm(x1, y1, 0x5410);
          o[3][tg] = __byte_perm(x1, y1, 0x7632);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(dst + (size_t)(4 * d4 + j) * kTok) = make_uint4(o[j][0], o[j][1], o[j][2], o[j][3]);
      }
      // the staged codes were written through the generic proxy; the slot's
      // next bulk copy (async proxy) must land after them
      fence_async_smem();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_n(&freeb[s], hp == 0 ? 1 + kNCW - nh : 1);
    advance(nh);
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

int largest_divisor_at_most(int n, int cap) {
  for (int d = n < cap ? n : cap; d > 1; --d)
    if (n % d == 0) return d;
  return 1;
}

ProdGeo producer_geo(const ProducerParams& p, bool fused) {
  ProdGeo g{};
  const int D = p.D, mh = 1024 / D;  // heads per unit: token rows of at most 2 KB
  const bool has_q = p.q != nullptr && p.Hq > 0;
  g.kvh = largest_divisor_at_most(p.Hkv, mh);
  g.qh = has_q ? largest_divisor_at_most(p.Hq, mh) : 1;
  g.nkv = p.Hkv / g.kvh;
  g.nq = has_q ? p.Hq / g.qh : 0;
  g.upt = 2 * g.nkv + g.nq;
  g.units = (long long)((p.T + kTok - 1) / kTok) * g.upt;
  g.row_stride = (g.kvh > g.qh ? g.kvh : g.qh) * D * 2 + 16;
  g.slot_bytes = kTok * g.row_stride;
  const int vpw = 32 / (D / 32), runs = D / 16;
  int off = 0;
  g.off_nscr = off;
  off += fused ? kNCW * vpw * (runs + 4) * 4 : 0;
  g.off_meta = off;
  off += kTR * (int)sizeof(TileMeta);
  g.off_cs = off;
  off += (fused && p.rd > 0) ? kTR * kTok * (p.rd + 4) * 4 : 0;
  g.off_sm = off;
  off += (fused && p.k_smooth) ? 2 * p.Hkv * D * 4 : 0;
  g.off_w = off;
  off += fused ? 2 * D * 4 : 0;
  g.off_bar = off;
  off += (2 * kMaxSlots + 2 * kTR) * 8 + 16 + kMaxSlots * 4;  // barriers, the abort flag, the slot stamps
  off = (off + 1023) & ~1023;
  int S = (kMaxSmem - off) / g.slot_bytes;
  if (S > kMaxSlots) S = kMaxSlots;
  g.S = S;
  // the ring first, the fixed regions after it
  const int ring = S * g.slot_bytes;
  g.off_nscr += ring;
  g.off_meta += ring;
  g.off_cs += ring;
  g.off_sm += ring;
  g.off_w += ring;
  g.off_bar += ring;
  g.smem = ring + off;
  return g;
}

int g_prod_sms[64] = {0};

int producer_sms(int device) {
  if (device < 0 || device >= 64) return 148;
  if (g_prod_sms[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0) n = 148;
    g_prod_sms[device] = n;
  }
  return g_prod_sms[device];
}

template <int D, bool kFused>
cudaError_t launch_producer_d(const ProducerParams& p, cudaStream_t stream) {
  const ProdGeo g = producer_geo(p, kFused);
  if (g.units == 0) return cudaSuccess;
  if (g.S < 2) return cudaErrorInvalidConfiguration;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // the shared-memory opt-in, once per device; setting it twice is harmless
  static bool opted_in[64] = {};
  const bool track = dev >= 0 && dev < 64;
  if (!track || !opted_in[dev]) {
    e = cudaFuncSetAttribute(kv_quant_write_kernel<D, kFused>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e != cudaSuccess) return e;
    if (track) opted_in[dev] = true;
  }
  const long long sms = producer_sms(dev);
  const int grid = (int)(g.units < sms ? g.units : sms);
  return launch_pdl(kv_quant_write_kernel<D, kFused>, dim3(grid), dim3(kProdThreads), (size_t)g.smem, stream, p, g);
}

}  // namespace

I8KV_DEFINE_ERROR_ACCESSOR(read_error_producer)

cudaError_t launch_kv_quant_write(const ProducerParams& p, cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  return p.D == 256 ? launch_producer_d<256, false>(p, stream) : launch_producer_d<128, false>(p, stream);
}

cudaError_t launch_kv_rope_quant_write(const ProducerParams& p, cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  return p.D == 256 ? launch_producer_d<256, true>(p, stream) : launch_producer_d<128, true>(p, stream);
}

cudaError_t launch_bf16_kv_write(const ProducerParams& p, uint16_t* k_cache, uint16_t* v_cache, cudaStream_t stream) {
  const long long total = (long long)p.T * p.Hkv * (p.D / 8);
  if (total == 0) return cudaSuccess;
  const int grid = (int)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
  bf16_kv_write_kernel<<<grid, 256, 0, stream>>>(p, k_cache, v_cache);
  return cudaGetLastError();
}

}  // namespace i8kv
