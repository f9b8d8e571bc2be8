/*
 * i8kv.h -- C ABI of the INT8 KV-cache paged-attention library for GB300 (sm_103a).
 *
 * The operation is the one described in two pages of a blog series:
 *   [KV] "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化" (part 1)
 *   [PV] "gfx936 DCU上实现INT8 PV MMAC：V Scale融合、概率量化与Fragment分组" (part 3)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers are DEVICE pointers unless a parameter says otherwise.  The caller
 *    owns every buffer; the library allocates nothing and keeps no state besides
 *    a per-thread last-error string and one device-side error word.
 *  - bf16 tensors are passed as `const uint16_t*` (raw bf16 bit patterns).
 *  - All launches are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL is the legacy default stream).  Nothing synchronizes.  Kernels are
 *    launched with programmatic dependent launch: a kernel may be scheduled
 *    while the previous kernel on the stream is still running, but it reads
 *    no global memory before that kernel has finished -- with one exception:
 *    the decode kernels read seq_lens and block_tables early (no kernel of
 *    this library writes them), so these two inputs must not be written by a
 *    kernel that may still be running when the decode call starts: the kernel
 *    launched just before it on the same stream, and any kernel before that
 *    one which let its successor start early (the decode merge kernels do so
 *    at their start, so a decode call may start while the previous call's
 *    attention kernel still runs; that kernel does not write them).  A host
 *    copy, or a kernel that completed before, is fine.  The decode kernels read them again after the wait and record
 *    error 3 in the device error word if they changed.
 *  - Argument errors are reported synchronously through the status code, before
 *    anything is launched; i8kv_last_error() gives a one-line reason.  A launch
 *    failure reported by the CUDA runtime maps to I8KV_ERR_CUDA.
 *  - Inputs are never written.  Outputs are fully overwritten.
 *  - Paged layouts ([KV] §2.3), with bs = block_size (16 is the only size the
 *    kernels accept), NB blocks in the pool, Hkv KV heads and head_dim D:
 *        K cache   int8  [NB, Hkv, D/16, bs, 16]   16 head-dims per 16-byte chunk
 *        V cache   int8  [NB, Hkv, D, bs]          tokens inner-most
 *        K/V scale fp32  [NB, bs, Hkv]             one scale per (token, KV head)
 *    A token at slot s lives in block s / bs at offset s % bs.  A sequence's
 *    token at position p lives in block block_table[p / bs], offset p % bs.
 *  - Cache, scale, Q and workspace pointers must be 16-byte aligned.
 *  - num_blocks is the pool size (blocks).  Kernels that read the cache check
 *    every block-table entry against it: an entry outside [0, num_blocks) is
 *    not read, the result is undefined, and the device error word records 2.
 *    A sequence length above max_blocks * block_size is clamped and recorded
 *    the same way.  Host-side checks cannot see device data, so these are the
 *    only checks on table contents.
 *  - Supported shapes: D in {128, 256}; Hq % Hkv == 0 with G = Hq / Hkv <= 8;
 *    query head h reads KV head h / G.
 *  - Quantization is symmetric INT8 with an fp32 absmax/127 scale per (token,
 *    head) vector; codes are clamp(round_half_even(x / scale), -127, 127); a
 *    vector of zeros gets scale 0 and zero codes ([KV] §2.1).
 */
#ifndef I8KV_H_
#define I8KV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  I8KV_OK = 0,
  I8KV_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer            */
  I8KV_ERR_UNSUPPORTED = 2, /* valid but not implemented (D, G, block size, partition) */
  I8KV_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required           */
  I8KV_ERR_CUDA = 4,        /* the CUDA runtime reported an error at launch         */
  I8KV_ERR_DEVICE = 5       /* a kernel recorded a failure in the device error word */
} i8kv_status;

/* Element type of an attention output ([KV] §3.3: the decode merges its      */
/* partitions and writes BF16).  I8KV_OUT_F32: fp32.  I8KV_OUT_BF16: the same  */
/* fp32 results rounded to nearest-even bf16 (raw bit patterns), half the     */
/* bytes.  Every attention entry point takes `void* out, int out_dtype`.      */
typedef enum { I8KV_OUT_F32 = 0, I8KV_OUT_BF16 = 1 } i8kv_out_dtype;

/* One-line description of the last non-OK status returned on this host thread.
 * Copies at most n-1 bytes plus a terminating NUL into buf (host memory). */
i8kv_status i8kv_last_error(char* buf, size_t n);

/* Reads and clears the device error word (synchronizes the device).  *code is
 * 0 when no kernel recorded a failure; otherwise the first failure's code:
 * 1 = a pipeline wait exceeded its time limit, 2 = a block-table or slot entry
 * or sequence length out of range (the access was skipped), 3 = seq_lens or
 * block_tables changed while a decode kernel was starting (they were written
 * by the kernel just before it on the stream; the result is undefined), 4 = a
 * RoPE position outside the cos/sin table (the token was skipped).  Returns
 * I8KV_ERR_DEVICE if *code != 0. */
i8kv_status i8kv_device_error(int* code);

/* Library version (major * 10000 + minor * 100 + patch). */
int i8kv_version(void);

/* ------------------------------------------------------------------------ */
/* KV producer ([KV] §2.2 "fused KV producer", steps 3-6, without RoPE).     */
/* For every token t < T with slot_mapping[t] >= 0 and every KV head h:      */
/*   quantize k[t,h,:] and v[t,h,:] (bf16 [T, Hkv, D]) per the rule above,   */
/*   store the codes at slot_mapping[t] in k_cache / v_cache and the scales  */
/*   in k_scale / v_scale.                                                   */
/* When q != NULL also quantize q (bf16 [T, Hq, D]) per (token, q-head) into */
/*   q_i8 (int8 [T, Hq, D]) and q_scale (fp32 [T, Hq]) -- the query is       */
/*   quantized once and reused by every history partition ([KV] §2.2).       */
/* Slots must lie inside the pool (num_blocks * block_size); two tokens with */
/* the same slot race.  A slot >= num_blocks * block_size is skipped and    */
/* recorded in the device error word (2).  slot < 0 skips only the K/V      */
/* write; the query row is still quantized.                                 */
/* The output codes and scales are bit-exact with the                       */
/* fp32 IEEE evaluation of the formula (division, not reciprocal).           */
/* ------------------------------------------------------------------------ */
i8kv_status i8kv_kv_quant_write(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping, int T, int Hkv,
                                int D, int block_size, int num_blocks, int8_t* k_cache, int8_t* v_cache,
                                float* k_scale, float* v_scale, const uint16_t* q, int Hq, int8_t* q_i8,
                                float* q_scale, void* stream);

/* ------------------------------------------------------------------------ */
/* Fused KV producer with Q/K RMSNorm and RoPE ([KV] §2.2 steps 1-6: RoPE on */
/* Q and K ahead of the absmax and the quantization; [KV] §5.3: the per-head */
/* Q/K RMSNorm that precedes RoPE).  Same outputs, rules and error handling  */
/* as i8kv_kv_quant_write, except that every Q and K vector x (bf16 -> fp32) */
/* is first transformed in fp32, each step one correctly rounded operation   */
/* in this order (no FMA contraction), so results are bit-reproducible:      */
/*   RMSNorm (when the kind's weight is given, bf16 [D]):                    */
/*     ss  = sum of x_i^2 as a balanced binary tree in index order           */
/*           (pairs (0,1), (2,3), ..., then pairs of those, ...);             */
/*     inv = 1 / sqrt(ss * (1/D) + norm_eps);   x_i = (x_i * inv) * w_i.      */
/*   RoPE, rotate-half on the first rotary_dim dims (h = rotary_dim / 2),    */
/*     with row r = cos_sin[positions[t]] (fp32 [max_position, rotary_dim]:  */
/*     cos of the h frequencies, then their sin):                            */
/*     a = x_i, b = x_{i+h}:  x_i = a*r[i] - b*r[h+i],  x_{i+h} = b*r[i] + a*r[h+i]*/
/*     (products rounded, then the sum).  Dims >= rotary_dim are unchanged.   */
/*   V is not transformed.                                                   */
/* rotary_dim: 0 (no RoPE; positions and cos_sin may be NULL) or a multiple  */
/*   of 32 up to D.  q_norm_weight / k_norm_weight: NULL skips that norm     */
/*   (q_norm_weight is ignored without q); norm_eps > 0 when either is given.*/
/* q_i8 / q_scale may both be NULL when q_out is given.                      */
/* q_out (bf16 [T, Hq, D]) and k_out (bf16 [T, Hkv, D]), nullable, receive   */
/*   the transformed Q / K rounded to nearest-even bf16, for every token     */
/*   whatever its slot (k_out lets a high-precision path reuse the rotated K).*/
/* A token whose position lies outside [0, max_position) is skipped entirely */
/*   (none of its outputs is written) and the device error word records 4.   */
/* k_smooth (fp32 [Hkv, D], nullable, entries > 0 and finite): per-channel   */
/*   K smoothing for stable channel outliers (KIVI's observation, cited in   */
/*   [KV] §2.1).  After RMSNorm and RoPE, K of KV head h is multiplied by    */
/*   RN(1/s[h][d]) and Q of query head hq by s[hq / G][d] (G = Hq / Hkv),    */
/*   each product rounded once; q.k is unchanged in exact arithmetic (the    */
/*   folding [PV] applies to sV), so the attention kernels need no change.   */
/*   q_out / k_out are taken before the smoothing.                           */
/* cos_sin, the norm weights and k_smooth must be 16-byte aligned.           */
/* ------------------------------------------------------------------------ */
i8kv_status i8kv_kv_rope_quant_write(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping, int T,
                                     int Hkv, int D, int block_size, int num_blocks, int8_t* k_cache, int8_t* v_cache,
                                     float* k_scale, float* v_scale, const uint16_t* q, int Hq, int8_t* q_i8,
                                     float* q_scale, const int32_t* positions, const float* cos_sin, int max_position,
                                     int rotary_dim, const uint16_t* q_norm_weight, const uint16_t* k_norm_weight,
                                     float norm_eps, uint16_t* q_out, uint16_t* k_out, const float* k_smooth,
                                     void* stream);

/* ------------------------------------------------------------------------ */
/* INT8 paged decode attention ([PV] §2-§3, [KV] §3.3).                     */
/* For sequence b (history L = seq_lens[b], every cached token 0..L-1) and   */
/* query head h (int8 q_i8[b,h,:] with scale q_scale[b,h]):                  */
/*   score_t = acc_t * sQ * sK_t * softmax_scale, acc_t = sum_d q*k (int32);  */
/*   history is cut into partitions of `partition` tokens; in partition g:    */
/*   m_g = max score, l_g = sum exp(score - m_g), P_t = exp(score_t - m_g)/l_g,*/
/*   W_t = P_t * sV_t; every 32-token group (aligned to position 0) of one   */
/*   query row is quantized with sW = max W / 127, Wq = round(W / sW), and   */
/*   o_g += sW * (Wq x Vq) with an int32 contraction; partitions are merged   */
/*   by log-sum-exp: O = sum_g l_g e^(m_g-M) o_g / sum_g l_g e^(m_g-M).      */
/* out: [B, Hq, D] of out_dtype (fp32, or bf16 = RNE of the fp32 result),    */
/*   16-byte aligned.  seq_lens[b] == 0 gives a zero row.                     */
/* block_tables: int32 [B, max_blocks]; entries past ceil(L/bs) are unused.  */
/* softmax_scale <= 0 selects 1/sqrt(D).  partition must be 256.             */
/* workspace: device memory of at least i8kv_decode_workspace_bytes(...)     */
/*   bytes; it needs no initialization (every record the call reads is      */
/*   written earlier in the same call).  Reuse it for later calls on the     */
/*   same stream; calls that overlap in time need separate workspaces.       */
/* The call launches two kernels (the attention and a merge of the pairs    */
/* whose history spans several CTAs).                                       */
/* ------------------------------------------------------------------------ */
size_t i8kv_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int max_blocks, int block_size, int partition);

i8kv_status i8kv_int8_paged_decode_attn(void* out, int out_dtype, const int8_t* q_i8, const float* q_scale,
                                        const int8_t* k_cache,
                                        const int8_t* v_cache, const float* k_scale, const float* v_scale,
                                        const int32_t* block_tables, const int32_t* seq_lens, int B, int Hq, int Hkv,
                                        int D, int block_size, int max_blocks, int num_blocks, float softmax_scale,
                                        int partition, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* The same decode with UINT8 probability codes ([PV] §6 weighs them: the   */
/* weights W = P x sV are non-negative, so codes 0..255 carry one bit more   */
/* than the signed 0..127; the pages leave the variant for want of a         */
/* mixed-sign MMA).  Per 32-token group sW = fp32(A / 255) and              */
/* Wq = round-half-even(W / sW) in 0..255; PV = Wq x Vq on the s8 x u8 MMA   */
/* (exact int32).  Arguments, layouts and workspace as above.                */
/* ------------------------------------------------------------------------ */
i8kv_status i8kv_int8_paged_decode_attn_u8p(void* out, int out_dtype, const int8_t* q_i8, const float* q_scale,
                                            const int8_t* k_cache, const int8_t* v_cache, const float* k_scale,
                                            const float* v_scale, const int32_t* block_tables,
                                            const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int block_size,
                                            int max_blocks, int num_blocks, float softmax_scale, int partition,
                                            void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Allocation-free variant of i8kv_int8_paged_decode_attn.  The pages have   */
/* no counterpart: this entry point exists for callers that cannot allocate   */
/* device memory when they run a decode step -- for example a plugin inside  */
/* another inference runtime, or a server whose memory planner reserved all  */
/* device memory at start-up -- and so cannot provide a workspace.           */
/* Same arguments and result as i8kv_int8_paged_decode_attn with an fp32 out  */
/* and without the workspace: the merge scratch is a fixed 8 MiB array inside the library    */
/* (8,388,608 bytes; every GPU that loads the library holds it until the     */
/* process exits).  It calls no cudaMalloc or cudaFree.                      */
/* Limit: i8kv_decode_workspace_bytes(B, Hq, Hkv, D, ...) must not exceed     */
/* 8 MiB (about (B*Hkv + number of SMs) * (32*D + 64) bytes), else the call   */
/* returns I8KV_ERR_WORKSPACE and launches nothing.                          */
/* The scratch's device address belongs to the CUDA context that loaded the */
/* library's code: the first call in each context (the device's primary     */
/* context, or a context the caller made current) looks it up and caches it */
/* under that context's id, so make the first call in each context before   */
/* any stream capture.  A device reset destroys the primary context; the    */
/* first call after it looks the address up again, for the new context.     */
/* All calls share the one scratch area: calls                              */
/* that overlap on the GPU (other streams, other host threads) race and give */
/* wrong results -- serialize them, e.g. on one stream.                      */
/* ------------------------------------------------------------------------ */
i8kv_status i8kv_int8_paged_decode_attn_noalloc(float* out, const int8_t* q_i8, const float* q_scale,
                                                const int8_t* k_cache, const int8_t* v_cache, const float* k_scale,
                                                const float* v_scale, const int32_t* block_tables,
                                                const int32_t* seq_lens, int B, int Hq, int Hkv, int D,
                                                int block_size, int max_blocks, int num_blocks, float softmax_scale,
                                                int partition, void* stream);

/* ------------------------------------------------------------------------ */
/* INT8 decode step: i8kv_kv_quant_write of every sequence's newest token    */
/* followed by i8kv_int8_paged_decode_attn, in one attention launch (plus    */
/* the merge).  The pages run the fused producer and the attention as two    */
/* kernels ([KV] §2.2, §3.3); here the attention kernel also does the        */
/* producer's work for the one new token per sequence:                       */
/*   k_new, v_new: bf16 [B, Hkv, D], the K/V of position L - 1 of sequence b */
/*   (L = seq_lens[b], which counts the new token).  They are quantized by    */
/*   the producer's rule (the same codes and scales, bit for bit) and written */
/*   into k_cache / v_cache / k_scale / v_scale at that position's slot       */
/*   (block block_tables[b][(L-1)/16], offset (L-1) % 16); the attention      */
/*   uses them as well.                                                       */
/*   q: bf16 [B, Hq, D], quantized per (sequence, q-head) by the producer's  */
/*   rule inside the kernel (the int8 query is not written out).             */
/* Everything else as i8kv_int8_paged_decode_attn.  seq_lens[b] == 0 means  */
/* no new token: a zero row and no write.  The output and the cache equal    */
/* those of the two calls bit for bit.  q, k_new, v_new: 16-byte aligned.    */
/* ------------------------------------------------------------------------ */
i8kv_status i8kv_int8_decode_step(void* out, int out_dtype, const uint16_t* q, const uint16_t* k_new,
                                  const uint16_t* v_new,
                                  int8_t* k_cache, int8_t* v_cache, float* k_scale, float* v_scale,
                                  const int32_t* block_tables, const int32_t* seq_lens, int B, int Hq, int Hkv, int D,
                                  int block_size, int max_blocks, int num_blocks, float softmax_scale, int partition,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* INT8 prefix-prefill chunk ([PV] §2.1, [KV] §3.2): one online softmax over */
/* the cached history and the chunk itself.  Chunk query j (absolute         */
/* position history_len + j) attends to cache positions 0..history_len + j   */
/* of the sequence described by block_table (int32, covering at least        */
/* history_len + chunk_len positions); the chunk's own K/V must already be   */
/* in the cache (written by i8kv_kv_quant_write).  Running state (m, l, o):  */
/*   alpha = exp(m - m'), p~_t = exp(score_t - m'), W_t = p~_t * sV_t        */
/*   (unnormalized), per (query row, 32-token group) sW = max W / 127,       */
/*   Wq = round(W / sW), o = alpha o + sum sW (Wq x Vq), l = alpha l + sum p~,*/
/*   O = o / l.                                                               */
/* q_i8: int8 [chunk_len, Hq, D], q_scale: fp32 [chunk_len, Hq].             */
/* out: [chunk_len, Hq, D] of out_dtype, 16-byte aligned.                     */
/* softmax_scale <= 0 selects 1/sqrt(D).                                     */
/* workspace: device memory of at least i8kv_prefix_workspace_bytes(...)    */
/*   bytes, 16-byte aligned, no initialization needed.  The call first      */
/*   writes into it the sequence's K/V codes as f16 (exact) operand tiles,  */
/*   one per (KV head, 32-key group), then runs the attention from them;    */
/*   about 4.1 bytes per cached (token, KV head, head dim), plus room for   */
/*   the split row blocks' partial results (2 x #SM x 128 rows x (D + 4)    */
/*   fp32, #SM of the current device).  Calls that overlap in time need     */
/*   separate workspaces.                                                   */
/* The call launches two kernels (the tiles and the attention), and a third */
/* that merges partial results when the last wave of 128-row blocks is      */
/* split over its keys (more row blocks than SMs, not a multiple of them).  */
/* ------------------------------------------------------------------------ */
size_t i8kv_prefix_workspace_bytes(int history_len, int chunk_len, int Hkv, int D);

i8kv_status i8kv_int8_prefix_attn(void* out, int out_dtype, const int8_t* q_i8, const float* q_scale,
                                  const int8_t* k_cache,
                                  const int8_t* v_cache, const float* k_scale, const float* v_scale,
                                  const int32_t* block_table, int history_len, int chunk_len, int Hq, int Hkv, int D,
                                  int block_size, int num_blocks, float softmax_scale, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* High-precision chunk attention ([KV] §3.1: the first prefill chunk keeps  */
/* a high-precision attention while the producer writes its K/V as INT8;     */
/* [KV] §4: below the routing threshold chunks stay high-precision).  Query  */
/* row j of the chunk (bf16 q [C, Hq, D], position history_len + j) attends  */
/* to keys 0 .. history_len + j:                                             */
/*   a history key t < history_len is read back from the INT8 cache as       */
/*   bf16(code x scale) (the cache keeps no other copy), through block_table */
/*   (entries for positions < history_len);                                  */
/*   a chunk key comes from the chunk's own bf16 k_chunk / v_chunk           */
/*   [C, Hkv, D], as given.                                                  */
/* S = Q K^T on bf16 tensor-core MMAs with fp32 accumulation; online softmax */
/* in fp32 over 32-key groups; P = p~ rounded to bf16 for the P V MMA; the   */
/* row sums l use the fp32 p~.  out: [C, Hq, D] of out_dtype.                */
/* history_len == 0 (a first chunk): the cache pointers, block_table and     */
/* num_blocks are not used and may be NULL / 0.                              */
/* workspace: as for i8kv_int8_prefix_attn (same size function; the tiles    */
/*   hold bf16 values instead of f16 codes).  Launches two kernels.          */
/* ------------------------------------------------------------------------ */
i8kv_status i8kv_bf16_prefix_attn(void* out, int out_dtype, const uint16_t* q, const uint16_t* k_chunk,
                                  const uint16_t* v_chunk,
                                  const int8_t* k_cache, const int8_t* v_cache, const float* k_scale,
                                  const float* v_scale, const int32_t* block_table, int history_len, int chunk_len,
                                  int Hq, int Hkv, int D, int block_size, int num_blocks, float softmax_scale,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* One prefill chunk, routed ([KV] §3.1-§3.2 and §4: the first chunk on the  */
/* high-precision attention, later chunks -- once the history reaches the    */
/* threshold -- wholly INT8, history and chunk in one online softmax).       */
/* Always: i8kv_kv_quant_write of the chunk's bf16 k, v [C, Hkv, D] to their */
/* slots (slot_mapping [C]), so the INT8 cache holds the chunk afterwards.   */
/* Then, with history_len >= int8_min_history: the query is quantized by the */
/* same call into q_i8 [C, Hq, D] / q_scale [C, Hq] (caller-owned scratch)   */
/* and i8kv_int8_prefix_attn runs over history + chunk; otherwise            */
/* i8kv_bf16_prefix_attn runs on the bf16 q, k, v (q_i8 / q_scale unused and */
/* may be NULL).  int8_min_history = 4096 is the pages' routing; 0 sends     */
/* every chunk to INT8, INT_MAX none.  block_table must cover history_len +  */
/* chunk_len positions.  *route (host int, nullable) receives the route      */
/* taken.  Inputs are assumed rotated already (i8kv_kv_rope_quant_write with */
/* q_out / k_out produces them).  Three launches: producer, tiles, attention.*/
/* ------------------------------------------------------------------------ */
#define I8KV_ROUTE_BF16 0
#define I8KV_ROUTE_INT8 1
i8kv_status i8kv_prefill_chunk(void* out, int out_dtype, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const int32_t* slot_mapping, int8_t* k_cache, int8_t* v_cache, float* k_scale,
                               float* v_scale, const int32_t* block_table, int history_len, int chunk_len, int Hq,
                               int Hkv, int D, int block_size, int num_blocks, int int8_min_history,
                               float softmax_scale, int8_t* q_i8, float* q_scale, void* workspace,
                               size_t workspace_bytes, int* route, void* stream);

/* ------------------------------------------------------------------------ */
/* Debug: raw int32 QK accumulators acc[b, h, t] = sum_d q_i8[b,h,d] *        */
/* K_i8[b, t, h / G, d] for t < seq_lens[b]; 0 for t in [seq_lens[b],        */
/* max_len).  Uses the decode kernel's paged-K addressing and MMA fragments, */
/* so a bit-exact match validates both ([PV] §2: the int32 accumulator).     */
/* acc: int32 [B, Hq, max_len].                                              */
/* ------------------------------------------------------------------------ */
i8kv_status i8kv_debug_qk_i32(int32_t* acc, const int8_t* q_i8, const int8_t* k_cache, const int32_t* block_tables,
                              const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int block_size, int max_blocks,
                              int num_blocks, int max_len, void* stream);

/* ------------------------------------------------------------------------ */
/* Debug: the prefix kernel's raw integer contractions ([PV] §3: INT8 Wq x   */
/* Vq accumulated in int32, at most 32 x 127 x 127 per group; [PV] §2: INT8  */
/* QK in int32).  Runs i8kv_int8_prefix_attn's kernels -- the same operand   */
/* tiles, tensor-core descriptors and tensor-memory reads -- on the same     */
/* arguments, writes the same fp32 out, and also records, for chunk row j    */
/* (position H + j) and query head h, with NG = ceil((H + C) / 32):         */
/*   s_acc  int32 [C, Hq, H + C]: S[t] = sum_d q_i8 * K_code[t] for every    */
/*          visible key t <= H + j, 0 for the others;                        */
/*   wq     uint8 [C, Hq, NG * 32]: the probability code Wq of each visible  */
/*          key (0..127), 0 for the others;                                  */
/*   pv_acc int32 [C, Hq, NG, D]: per 32-key group g the contraction         */
/*          sum_{t in g} Wq[t] * V_code[t][d] as the kernel read it from     */
/*          tensor memory; 0 for groups the row's block never reaches.       */
/* The records are cleared on the stream first (cudaMemsetAsync).  Meant for */
/* tests: the stores make it slow.                                          */
/* ------------------------------------------------------------------------ */
i8kv_status i8kv_debug_prefix_i32(int32_t* s_acc, uint8_t* wq, int32_t* pv_acc, float* out, const int8_t* q_i8,
                                  const float* q_scale, const int8_t* k_cache, const int8_t* v_cache,
                                  const float* k_scale, const float* v_scale, const int32_t* block_table,
                                  int history_len, int chunk_len, int Hq, int Hkv, int D, int block_size,
                                  int num_blocks, float softmax_scale, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* ------------------------------------------------------------------------ */
/* BF16-KV comparison path (the pages' BF16 control: same paging, bf16      */
/* elements, bf16 tensor-core contractions, fp32 softmax; [KV] §4.2).       */
/*   K cache bf16 [NB, Hkv, D/8, bs, 8], V cache bf16 [NB, Hkv, D, bs].      */
/* ------------------------------------------------------------------------ */
i8kv_status i8kv_bf16_kv_write(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping, int T, int Hkv,
                               int D, int block_size, int num_blocks, uint16_t* k_cache, uint16_t* v_cache,
                               void* stream);

/* The prefix chunk over the bf16 cache (the BF16 control of the pages'      */
/* prefill comparison, [KV] §4.2): chunk row j (bf16 q [C, Hq, D], position   */
/* history_len + j) attends to keys 0 .. history_len + j of the sequence,    */
/* every key -- history and the chunk's own, which must already be in the    */
/* cache (i8kv_bf16_kv_write) -- read from the bf16 cache through            */
/* block_table.  The kernels are those of i8kv_bf16_prefix_attn (bf16        */
/* tensor-core MMAs, fp32 online softmax over 32-key groups, p~ rounded to   */
/* bf16 for P x V, fp32 row sums) with operand tiles built from the bf16     */
/* cache.  out: [C, Hq, D] of out_dtype.  workspace: as for                  */
/* i8kv_int8_prefix_attn (same size function).  Launches two kernels (three  */
/* with a split last wave).                                                  */
i8kv_status i8kv_bf16_kv_prefix_attn(void* out, int out_dtype, const uint16_t* q, const uint16_t* k_cache,
                                     const uint16_t* v_cache, const int32_t* block_table, int history_len,
                                     int chunk_len, int Hq, int Hkv, int D, int block_size, int num_blocks,
                                     float softmax_scale, void* workspace, size_t workspace_bytes, void* stream);

/* Plain softmax decode attention over the bf16 cache with the same 256-token
 * partitions and log-sum-exp merge.  q: bf16 [B, Hq, D]; out: [B, Hq, D] of
 * out_dtype.
 * The workspace follows the same rules and size as the INT8 decode's. */
i8kv_status i8kv_bf16_paged_decode_attn(void* out, int out_dtype, const uint16_t* q, const uint16_t* k_cache,
                                        const uint16_t* v_cache, const int32_t* block_tables,
                                        const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int block_size,
                                        int max_blocks, int num_blocks, float softmax_scale, int partition,
                                        void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* I8KV_H_ */
