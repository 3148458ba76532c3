/*
 * pva.h -- packed varlen (document-masked) attention on one GB300 (sm_103a).
 *
 * C ABI.  Every pointer is either a HOST pointer or a DEVICE pointer, as
 * stated per argument.  The caller allocates and owns every buffer (the
 * library allocates no memory); device work is enqueued on the caller's
 * CUDA stream (`stream` is a cudaStream_t, NULL = legacy default stream) and
 * is asynchronous.  Argument errors are detected on the host and returned
 * before anything is enqueued.  A launch failure returns PVA_ERR_CUDA.
 * Device-side failures (a bounded wait that timed out, a worklist that does
 * not match the call) are recorded in the worklist's error word and read
 * with pva_worklist_error().
 *
 * The method is the hot path of the long-context load-balancing pages:
 *  - "03 · 长文负载均衡" §1.1: documents packed into one sequence attend only
 *    to themselves, so a pack's attention work is sum_j l_j^2, not
 *    (sum_j l_j)^2; THD packing with cu_seqlens (§2.4).
 *  - §1.2: structured masks (sliding window, shared question).
 *  - §3.2: tiles charged by their exact causal query-key pair count (Libra
 *    TAP); a computation block exists only where the mask is non-zero (DCP).
 *  - §2.1 and "数据并行负载均衡" §4.4: LPT (longest processing time first)
 *    placement, here over the persistent CTAs of one GPU.
 *  - §4.2-4.3: zigzag context parallelism, per document.
 *  - §3.2 and the ring-attention notes of "长序列训练与上下文并行": partial
 *    (O, LSE) results merged by online softmax.
 *
 * Layouts (all row-major, contiguous, 16-byte aligned):
 *   Q     [q_tokens, num_q_heads,  head_dim]  bf16
 *   K, V  [k_tokens, num_kv_heads, head_dim]  bf16
 *   O     [q_tokens, num_q_heads,  head_dim]  bf16, or fp32 for partials
 *   LSE   [num_q_heads, q_tokens]             fp32, natural log
 *   cu_seqlens int32 [num_docs + 1], 0 = cu[0] <= cu[1] <= ... (empty docs allowed)
 * GQA: q head h reads kv head h / (num_q_heads / num_kv_heads).
 * Rows with no allowed key produce O = 0 and LSE = -inf.
 */
#ifndef PVA_H
#define PVA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PVA_OK = 0,
    PVA_ERR_INVALID_ARG = 1,      /* bad size, pointer, alignment or mask field */
    PVA_ERR_BUFFER_TOO_SMALL = 2, /* worklist buffer smaller than pva_worklist_bytes() */
    PVA_ERR_CUDA = 3,             /* a CUDA runtime/driver call failed */
    PVA_ERR_UNSUPPORTED = 4,      /* valid but not implemented (head_dim, tiles) */
    PVA_ERR_TIMEOUT = 5,          /* a device-side bounded wait expired */
    PVA_ERR_DEVICE = 6            /* device-side consistency check failed */
} pva_status;

/* Mask kinds ("03 · 长文负载均衡" §1.1, §1.2, §4.2-4.4). */
typedef enum {
    PVA_MASK_CAUSAL = 0,          /* per document: k <= q */
    PVA_MASK_SLIDING_WINDOW = 1,  /* per document: k <= q and q - k < window */
    PVA_MASK_SHARED_QUESTION = 2, /* docs [0, num_prefix_docs) are questions (causal on
                                     themselves); every later doc sees all question
                                     tokens and itself causally */
    PVA_MASK_ZIGZAG_PAIR = 3,     /* Q = zigzag shard of q_rank, K/V = shard of k_rank
                                     (rows in pva_zigzag_shard order); same document and
                                     k position <= q position */
    PVA_MASK_SLICES = 4,          /* explicit slice list (AttnSlice, §4.4) */
    PVA_MASK_ZIGZAG_STEP = 5      /* one ring step of all cp zigzag ranks at once: Q, K and V
                                     in ring order (rank 0's shard rows, then rank 1's, ...;
                                     pva_zigzag_ring_map), the query rows of rank r see the
                                     key rows of rank (r - ring_step) mod cp under the
                                     ZIGZAG_PAIR rule; q_tokens = k_tokens = cu[num_docs] */
} pva_mask_kind;

/* The four MaskTypes of "03 · 长文负载均衡" §4.4 (the pages name them without
 * geometry; the tests below use token positions, like the per-document masks):
 *   FULL         every (query, key) pair of the rectangle
 *   CAUSAL       k_pos <= q_pos           (window w > 0: and q_pos - k_pos < w)
 *   INV_CAUSAL   k_pos >= q_pos           (window w > 0: and k_pos - q_pos < w)
 *   BI_CAUSAL    k_pos >= q_pos and k_end - k_pos >= q_end - q_pos, with
 *                q_end = q_pos0 + q_len, k_end = k_pos0 + k_len: inverse-causal
 *                from the slice's start and causal from its end (for q_pos0 =
 *                k_pos0 the band q_pos <= k_pos <= q_pos + k_len - q_len);
 *                window must be 0. */
typedef enum {
    PVA_SLICE_FULL = 0,
    PVA_SLICE_CAUSAL = 1,
    PVA_SLICE_INV_CAUSAL = 2,
    PVA_SLICE_BI_CAUSAL = 3
} pva_slice_type;

/* One AttnSlice ("03 · 长文负载均衡" §4.4: (QRange, KRange, MaskType)).
 * Rows are indices into the Q / K buffers; positions are the rows' token
 * positions used by the mask tests above.  Consecutive slices with the same
 * (q_row0, q_len, q_pos0) form one query segment; the query ranges of
 * different segments must not overlap.  Query rows outside every slice are
 * not written. */
typedef struct {
    int32_t q_row0, q_len, q_pos0;
    int32_t k_row0, k_len, k_pos0;
    int32_t type;   /* pva_slice_type */
    int32_t window; /* <= 0: no window */
} pva_slice;

typedef struct {
    int32_t kind;            /* pva_mask_kind */
    int32_t window;          /* SLIDING_WINDOW: window >= 1 */
    int32_t num_prefix_docs; /* SHARED_QUESTION */
    int32_t cp, q_rank, k_rank; /* ZIGZAG_PAIR: 0 <= ranks < cp */
    const pva_slice* slices;    /* SLICES: HOST array of num_slices entries */
    int32_t num_slices;
    int32_t q_tokens;        /* rows of Q / O (for ZIGZAG_PAIR: pva_zigzag_shard_len(q_rank)) */
    int32_t k_tokens;        /* rows of K / V */
    int32_t ring_step;       /* ZIGZAG_STEP (with cp): 0 <= ring_step < cp */
} pva_mask_desc;

/* Worklist parameters.  The attention kernel supports tile_m = tile_n = 128,
 * head_dim 64 or 128.  Work units pair two 128-row query sub-tiles that share
 * one kv head: two q heads of a GQA group on the same q tile, or (for a
 * group's odd last head, or MHA) two consecutive q tiles of one head. */
typedef struct {
    int32_t tile_m, tile_n;
    int32_t num_q_heads, num_kv_heads;
    int32_t num_ctas;   /* persistent CTAs (bins of the LPT); <= 0: number of SMs */
    int32_t refine_iters; /* move/swap rounds after LPT ("数据并行负载均衡" §4.4 phase 2):
                             the most and least loaded CTAs, stop under a 5% gap; the
                             better of moving the heavy CTA's costliest unit or swapping it
                             with the light CTA's cheapest one, if it shrinks their gap.
                             0: none.  At most 1000. */
    int64_t c_tile;     /* fixed cost, in pair units (>= 0), of one computed (sub-tile, kv
                           tile) and of one query sub-tile (Q load, output rows):
                           unit cost = exact allowed pairs
                                       + c_tile * (sub-tiles * kv tiles + sub-tiles) */
    int32_t dispatch;   /* pva_dispatch: how the forward kernel's CTAs take their units */
    int32_t pack_docs;  /* 1: short documents share tiles ("03 · 长文负载均衡" §4.1: a block
                           shorter than a tile is still charged as a whole tile).  CAUSAL and
                           SLIDING_WINDOW masks: consecutive documents shorter than tile_m are
                           grouped greedily, in order, into groups of at most tile_m rows; a
                           group of two or more non-empty documents is one query tile against
                           one key tile, each row masked to its own document.  Other mask kinds
                           ignore it.  0: every document has its own tiles. */
} pva_worklist_params;

/* How the forward kernel hands units to its persistent CTAs.  Both follow the
 * LPT rule of "数据并行负载均衡" §4.4 (units in decreasing cost, each to the
 * least loaded CTA).  The worklist is built for one of them and the forward
 * launch must name the same one (else the kernel reports a bad worklist).
 *   DYNAMIC (default): the builder also writes a dispatch order (power-of-two
 *     cost classes floor(log2(max(cost, 1))) in decreasing order, enumeration
 *     order inside a class, so that concurrent CTAs share the same documents'
 *     K/V in L2); a CTA that runs out of work claims the next unit of that
 *     order from a counter kept in the worklist, so "least loaded" is decided
 *     by measured time (list scheduling).  One worklist then serves one
 *     forward launch at a time (stream-ordered launches are fine); the last
 *     CTA to finish resets the counter.
 *   STATIC: each CTA runs the list the builder assigned it by cost (the exact
 *     LPT bins + refinement, the per-CTA CSR lists, enumeration order).
 * The per-CTA lists are built in both modes (the backward's dQ pass uses them). */
typedef enum {
    PVA_DISPATCH_DYNAMIC = 0,
    PVA_DISPATCH_STATIC = 1,
} pva_dispatch;

/* Upper bound, in bytes, of the device worklist for this problem.  HOST
 * computation only.  num_docs is the length of cu_seqlens minus one.
 * Returns 0 on invalid arguments. */
size_t pva_worklist_bytes(int32_t num_docs, const pva_mask_desc* mask,
                          const pva_worklist_params* params);

/* Build the worklist on the device ("03 · 长文负载均衡" §3.2, §2.1):
 * derive the slices of the mask, enumerate every (query sub-tile, kv tile)
 * work item with at least one allowed pair, cost each work unit by its exact
 * pair count (+ c_tile per tile and per sub-tile), then as params->dispatch
 * says: STATIC sorts by cost descending (stable) and assigns LPT-style to
 * params->num_ctas bins (lightest bin, lowest id on ties); DYNAMIC writes the
 * dispatch order the CTAs claim from at run time (pva_dispatch).
 *   cu_seqlens_dev  DEVICE int32 [num_docs + 1]
 *   worklist_dev    DEVICE buffer of worklist_bytes >= pva_worklist_bytes(), 256-B aligned
 * The result is deterministic and identical for identical inputs. */
pva_status pva_build_worklist(const int32_t* cu_seqlens_dev, int32_t num_docs,
                              const pva_mask_desc* mask, const pva_worklist_params* params,
                              void* worklist_dev, size_t worklist_bytes, void* stream);

/* Attention forward over the worklist: one persistent launch of
 * params->num_ctas CTAs (TMA-staged K/V tiles, tcgen05 MMAs into TMEM,
 * online softmax in fp32, masked tiles never visited).
 *   q, k, v         DEVICE bf16, layouts above; head_dim 64 or 128
 *   worklist_dev    DEVICE, built by pva_build_worklist with the same mask/params
 *   out             DEVICE, bf16 (out_is_fp32 = 0) or fp32 (out_is_fp32 = 1)
 *   lse             DEVICE fp32 [num_q_heads, q_tokens]
 *   softmax_scale   <= 0 selects 1/sqrt(head_dim)
 *   cta_busy_ns     DEVICE uint64 [num_ctas, 2] (start, end) globaltimer stamps, or NULL
 * cu_seqlens_dev and mask describe the same problem as the worklist and are
 * used only for argument checks.  With mask->q_tokens = 0 the call does nothing
 * and returns PVA_OK (q, k, v, out and lse may then be NULL). */
pva_status pva_attn_fwd(const void* q, const void* k, const void* v,
                        const int32_t* cu_seqlens_dev, const pva_mask_desc* mask,
                        const pva_worklist_params* params, int32_t head_dim,
                        const void* worklist_dev, void* out, int32_t out_is_fp32, float* lse,
                        float softmax_scale, uint64_t* cta_busy_ns, void* stream);

/* Fused ring step ("03 · 长文负载均衡" §3.2: DCP reduces partial outputs;
 * "长序列训练与上下文并行", ring attention: each step's local result is merged
 * into the running state).  Same arguments as pva_attn_fwd, except that the
 * output is a running pair that the call reads and updates in place:
 *   o_run    DEVICE fp32 [q_tokens, num_q_heads, head_dim]
 *   lse_run  DEVICE fp32 [num_q_heads, q_tokens]
 * For every query row with at least one allowed key in this call:
 *   lse' = ln(e^lse_run + e^lse_step),
 *   o'   = e^(lse_run - lse') o_run + e^(lse_step - lse') o_step
 * (o_run is not read where lse_run = -inf).  Rows with no allowed key in this
 * call keep their running values.  Start a ring with o_run = 0 and
 * lse_run = -inf (rows that never receive a key then end as O = 0,
 * LSE = -inf, as with separate partials and merges).  The
 * result equals pva_attn_fwd into fp32 partials followed by pva_merge_partials,
 * without the partial buffers or the separate merge pass. */
pva_status pva_attn_fwd_accumulate(const void* q, const void* k, const void* v,
                                   const int32_t* cu_seqlens_dev, const pva_mask_desc* mask,
                                   const pva_worklist_params* params, int32_t head_dim,
                                   const void* worklist_dev, float* o_run, float* lse_run,
                                   float softmax_scale, uint64_t* cta_busy_ns, void* stream);

/* Rows of zigzag shard `rank` ("03 · 长文负载均衡" §4.2-4.3): every document
 * is cut into 2*cp contiguous chunks, chunk c holding floor(l/2cp) tokens
 * plus one if c < l mod 2cp; rank r owns chunks r and 2cp-1-r of every
 * document.  HOST computation on a HOST cu_seqlens.  Returns -1 on bad input. */
int32_t pva_zigzag_shard_len(const int32_t* cu_seqlens_host, int32_t num_docs, int32_t cp,
                             int32_t rank);

/* Zigzag index maps on the device.
 *   cu_seqlens_dev   DEVICE int32 [num_docs + 1]
 *   gather_map_dev   DEVICE int32 [pva_zigzag_shard_len(...)]: local row -> global token;
 *                    per document, chunk r then chunk 2cp-1-r
 *   chunk_table_dev  DEVICE int32 [num_docs][2][4] (doc, chunk, global start, length), or NULL */
pva_status pva_zigzag_shard(const int32_t* cu_seqlens_dev, int32_t num_docs, int32_t cp,
                            int32_t rank, int32_t* gather_map_dev, int32_t* chunk_table_dev,
                            void* stream);

/* Ring order of all zigzag shards on the device ("长序列训练与上下文并行", ring
 * attention over cp ranks, each holding its zigzag shard): ring_map_dev[i] =
 * global token of row i of the concatenation of the shards of ranks 0, 1, ...,
 * cp-1, each in pva_zigzag_shard order (cu_seqlens[num_docs] entries).  Q, K
 * and V gathered through this map are the inputs of PVA_MASK_ZIGZAG_STEP.
 *   cu_seqlens_dev DEVICE int32 [num_docs + 1];  ring_map_dev DEVICE int32 */
pva_status pva_zigzag_ring_map(const int32_t* cu_seqlens_dev, int32_t num_docs, int32_t cp,
                               int32_t* ring_map_dev, void* stream);

/* Row gather for shard emulation: dst[i] = src[map[i]] for i < rows, rows of
 * row_bytes bytes (a multiple of 16); scatter = 1 writes dst[map[i]] = src[i].
 *   src, dst  DEVICE, 16-byte aligned;  map_dev DEVICE int32 [rows]
 *   indexed_rows  rows of the tensor that map[] indexes (src, or dst when
 *                 scattering); entries outside [0, indexed_rows) are skipped. */
pva_status pva_gather_rows(const void* src, const int32_t* map_dev, void* dst, int64_t rows,
                           int64_t row_bytes, int64_t indexed_rows, int32_t scatter,
                           void* stream);

/* Online-softmax merge of two partials over disjoint key sets
 * ("03 · 长文负载均衡" §3.2 DCP reduction; ring attention merge):
 *   lse = ln(e^{lse_a} + e^{lse_b}),  O = e^{lse_a - lse} O_a + e^{lse_b - lse} O_b
 * Both -inf gives O = 0, lse = -inf.  O_a, O_b, out: DEVICE [tokens, heads, head_dim]
 * fp32 (o_is_fp32 = 1) or bf16; lse_*: DEVICE fp32 [heads, tokens].  In place
 * (out == o_a, lse_out == lse_a) is allowed. */
pva_status pva_merge_partials(const void* o_a, const float* lse_a, const void* o_b,
                              const float* lse_b, void* out, float* lse_out, int64_t tokens,
                              int32_t heads, int32_t head_dim, int32_t o_is_fp32, void* stream);

/* ---- Backward ("03 · 长文负载均衡" §1.1: gradients of the QK^T and PV terms) ----
 * With P = exp(scale S - LSE) recomputed from the forward's LSE:
 *   dP = dO V^T, D = rowsum(dO * O), dS = P (dP - D),
 *   dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO (a kv head sums its group).
 * dQ runs over the forward worklist (same units and CTA lists); dK and dV run
 * over a backward plan of kv-major units: slices with the same key range form
 * a key group, and a unit is one 128-key tile of a group for one kv head,
 * covering every q tile of every slice of the group and every head of the kv
 * head's group that may see the tile's keys, accumulated in tensor memory
 * (each output row has one writer; results are deterministic).  Explicit
 * slices whose key ranges overlap without being equal, or more than 8192
 * slices, have no plan (0 bytes). */

/* Size of the backward plan (HOST computation; 0 if unsupported or invalid).
 * It also holds the D scratch, [num_q_heads, q_tokens] fp32. */
size_t pva_bwd_plan_bytes(int32_t num_docs, const pva_mask_desc* mask,
                          const pva_worklist_params* params);

/* Build the backward plan on the device from a built forward worklist of the
 * same problem: kv-major units and their cost (q-tile steps over the group's
 * heads + 1).  Under static dispatch they are sorted by cost descending and
 * the CTAs take them in snake order; under dynamic dispatch the CTAs claim
 * them by power-of-two cost class (descending), inside a class group by
 * group, kv head by kv head, key tiles ascending (concurrent units then read
 * the same documents' query tiles from L2).
 *   worklist_dev DEVICE (pva_build_worklist output);  plan_dev DEVICE, 256-B
 *   aligned, plan_bytes >= pva_bwd_plan_bytes() */
pva_status pva_build_bwd_plan(const void* worklist_dev, int32_t num_docs,
                              const pva_mask_desc* mask, const pva_worklist_params* params,
                              void* plan_dev, size_t plan_bytes, void* stream);

/* Attention backward over the forward worklist and the backward plan.
 *   q, k, v        DEVICE bf16, as for pva_attn_fwd
 *   out, lse       DEVICE: the forward's bf16 output and fp32 LSE [Hq, q_tokens]
 *   dout           DEVICE bf16 [q_tokens, Hq, head_dim]
 *   dq             DEVICE [q_tokens, Hq, head_dim], dk/dv DEVICE [k_tokens, Hkv,
 *                  head_dim]; bf16 (grads_are_fp32 = 0) or fp32 (= 1); written
 *                  (rows no slice reaches get 0)
 *   softmax_scale  <= 0 selects 1/sqrt(head_dim)
 * Four kernels on `stream` (D, dQ, dK/dV); device failures go to the forward
 * worklist's error word. */
pva_status pva_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, const int32_t* cu_seqlens_dev,
                        int32_t num_docs, const pva_mask_desc* mask,
                        const pva_worklist_params* params, int32_t head_dim,
                        const void* worklist_dev, void* plan_dev, void* dq, void* dk, void* dv,
                        int32_t grads_are_fp32, float softmax_scale, void* stream);

/* ---- Sharding solvers for context parallelism ("03 · 长文负载均衡" §4.2-§4.4) ----
 * They plan how the query rows of a pack are split over cp ranks; the pieces
 * then run through pva_build_worklist / pva_attn_fwd (e.g. as AttnSlices). */

/* Mask area of equal query chunks (§4.4, MagiAttention's dispatch input): the
 * pack's rows are cut into chunks of chunk_size rows (the last one possibly
 * shorter) and areas_dev[c] = allowed (query, key) pairs of chunk c's rows.
 * Mask kinds over the whole pack only: PVA_MASK_CAUSAL, _SLIDING_WINDOW,
 * _SHARED_QUESTION (mask->q_tokens = mask->k_tokens = cu_seqlens[num_docs]);
 * others return PVA_ERR_UNSUPPORTED.
 *   cu_seqlens_dev DEVICE int32 [num_docs + 1]
 *   areas_dev      DEVICE int64 [ceil(q_tokens / chunk_size)], written */
pva_status pva_chunk_areas(const int32_t* cu_seqlens_dev, int32_t num_docs,
                           const pva_mask_desc* mask, int32_t chunk_size, int64_t* areas_dev,
                           void* stream);

/* Greedy dispatch of num_chunks chunks into cp buckets of exactly
 * num_chunks / cp chunks each, minimising the largest bucket area (§4.4:
 * chunks by area descending, ties by lower chunk index; each to the bucket
 * with the smallest area that still has room, ties by lower bucket id).
 * num_chunks must be a multiple of cp; at most 8192 chunks and 1024 buckets
 * (PVA_ERR_UNSUPPORTED beyond).  One CTA; deterministic.
 *   areas_dev        DEVICE int64 [num_chunks] (>= 0)
 *   bucket_dev       DEVICE int32 [num_chunks], written: bucket of each chunk
 *   bucket_area_dev  DEVICE int64 [cp], written: area of each bucket */
pva_status pva_dispatch_chunks(const int64_t* areas_dev, int32_t num_chunks, int32_t cp,
                               int32_t* bucket_dev, int64_t* bucket_area_dev, void* stream);

/* Striped sharding (§4.2, Striped Attention: stripes of the whole sequence
 * interleaved across ranks): token i belongs to rank (i / stripe) mod cp.
 * _len is HOST computation (-1 on bad arguments); pva_striped_shard writes
 * rank's tokens in ascending order to map_dev (DEVICE int32 [len]). */
int32_t pva_striped_shard_len(int32_t total_tokens, int32_t cp, int32_t rank, int32_t stripe);
pva_status pva_striped_shard(int32_t total_tokens, int32_t cp, int32_t rank, int32_t stripe,
                             int32_t* map_dev, void* stream);

/* WLB-LLM's choice between per-sequence and per-document zigzag sharding of a
 * causal pack (§4.3): for each scheme, each of the cp workers' attention work
 * in tile-rounded FLOPs (a piece shorter than a tile is charged whole tiles:
 * q tiles of `tile` rows aligned at each piece start, ceil((P + 1) / tile) key
 * tiles for a q tile whose last document position is P, 4 * head_dim FLOPs
 * per pair of a computed tile).  Per-sequence cuts the whole pack into 2 cp
 * zigzag chunks (worker r: chunks r and 2cp - 1 - r), per-document cuts every
 * document that way.  HOST computation.
 *   cu_seqlens_host HOST int32 [num_docs + 1]
 *   costs_host      HOST int64 [2 * cp], written: per worker, per-sequence then
 *                   per-document
 * Returns 0 (per-sequence) or 1 (per-document): the scheme whose most loaded
 * worker is lighter (per-sequence on ties); -1 on bad arguments. */
int32_t pva_wlb_choose(const int32_t* cu_seqlens_host, int32_t num_docs, int32_t cp,
                       int32_t tile, int32_t head_dim, int64_t* costs_host);

/* Fitted per-tile cost ("数据并行负载均衡" §4.2: the load model's coefficients are
 * fitted to measured times during warm-up iterations, non-negative, with no
 * constant term).  From num_runs pva_attn_fwd runs, each over worklists_dev[r]
 * with cta_busy_ns recorded in cta_busy_ns_dev[r], every CTA that had work
 * gives one sample
 *   t_b = a * pairs_b + c * (tiles_b + subtiles_b),   a, c >= 0
 * (its summed allowed pairs, (sub-tile, kv tile) steps and query sub-tiles),
 * fitted by non-negative least squares over all samples.
 * A worklist balanced by LPT makes every CTA's cost about equal, so pool runs
 * whose worklists were built with different c_tile (e.g. 0 and a large one).
 *   worklists_dev    HOST array [num_runs] of DEVICE worklists
 *   cta_busy_ns_dev  HOST array [num_runs] of DEVICE uint64 [num_ctas, 2]
 *   c_tile_out       HOST: round(c / a) (at most 2^24; 2^24 when a = 0 < c: the
 *                    time follows tiles alone), for pva_worklist_params.c_tile
 *   coef_out         HOST double [2] {a ns per pair, c ns per tile}, or NULL
 * Copies the worklists' units to the host and synchronizes `stream`.
 * The worklists must be built for PVA_DISPATCH_STATIC (per-CTA samples need
 * the static assignment); PVA_ERR_INVALID_ARG otherwise, and if both
 * coefficients are zero (no usable sample). */
pva_status pva_fit_tile_cost(const void* const* worklists_dev,
                             const uint64_t* const* cta_busy_ns_dev, int32_t num_runs,
                             int64_t* c_tile_out, double* coef_out, void* stream);

/* Device error word of a worklist (0 = none; otherwise the failing wait site,
 * see PVA_ERR_TIMEOUT / PVA_ERR_DEVICE).  Synchronizes `stream`.
 *   worklist_dev DEVICE;  code_out HOST */
pva_status pva_worklist_error(const void* worklist_dev, int32_t* code_out, void* stream);

/* Summary counts of a built worklist (HOST out, synchronizes `stream`):
 * out[0] segments, [1] slices, [2] units, [3] runs, [4] allowed pairs per head,
 * [5] kv tiles computed per head, [6] parallel steps the LPT took. */
pva_status pva_worklist_counts(const void* worklist_dev, int64_t* out7, void* stream);

/* Worklist build + attention forward for callers that cannot allocate device
 * memory (a plugin in a runtime that owns a fixed memory pool, a serving
 * process with a memory budget fixed up front, a C host without a device
 * allocator).  The pages have no counterpart: this is a packaging variant of
 * pva_build_worklist + pva_attn_fwd.  The caller passes inputs and outputs
 * only (same meaning as there; cta_busy_ns is not recorded); the worklist
 * lives in a static device array of pva_noalloc_scratch_bytes() (16 MiB) that
 * every GPU loading the library holds until the process exits.
 *  - Problems whose worklist (pva_worklist_bytes) exceeds that size are
 *    rejected with PVA_ERR_BUFFER_TOO_SMALL before any device work.
 *  - The first call on each device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *    Under CUDA's lazy module loading (the default) that first lookup is also
 *    when the driver loads the module and commits the 16 MiB on the device, so
 *    a caller with a fixed memory budget makes one warm-up call at start-up,
 *    before it fixes the budget.  The address is cached per device and per
 *    CUDA context (a new context, e.g. after cudaDeviceReset, is looked up
 *    again).
 *  - All calls on a device share the array, which keeps the last call's
 *    contents (the build rewrites everything it reads); calls that overlap on
 *    the GPU race on it.
 *  - Device-side failures (cu_seqlens that do not match the mask, a capacity
 *    overflow, a bounded wait that expired) leave out / lse unwritten and are
 *    recorded in the array's error word: read it with pva_noalloc_error().
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
pva_status pva_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                const int32_t* cu_seqlens_dev, int32_t num_docs,
                                const pva_mask_desc* mask, const pva_worklist_params* params,
                                int32_t head_dim, void* out, int32_t out_is_fp32, float* lse,
                                float softmax_scale, void* stream);

/* One forward pass for a caller whose inputs and results are in HOST memory
 * ("03 · 长文负载均衡" §1.1: the packed pack's attention).  Enqueued on
 * `stream`, in order: the copies of Q, K, V and cu_seqlens to the caller's
 * device buffers (one cudaMemcpyAsync each), pva_build_worklist,
 * pva_attn_fwd (bf16 output), and the copies of O and LSE back to the host.
 *   q_host, k_host, v_host   HOST bf16, the pva_attn_fwd layouts
 *   cu_seqlens_host          HOST int32 [num_docs + 1] (unused for PVA_MASK_SLICES)
 *   out_host                 HOST bf16 [q_tokens, num_q_heads, head_dim]
 *   lse_host                 HOST fp32 [num_q_heads, q_tokens]
 *   q_dev .. lse_dev         DEVICE buffers of the same sizes (caller-owned),
 *                            worklist_dev of worklist_bytes (as for pva_build_worklist)
 * The host buffers should be page-locked: with pageable memory the copies
 * still happen, but the call then waits for them.  The call returns once
 * everything is enqueued; the results are in out_host / lse_host when the
 * stream reaches this point.  Device-side failures go to the worklist's error
 * word.  Callers streaming packs alternate two streams and two sets of device
 * buffers, so that one pack's copies overlap the previous pack's attention. */
pva_status pva_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                             const int32_t* cu_seqlens_host, int32_t num_docs,
                             const pva_mask_desc* mask, const pva_worklist_params* params,
                             int32_t head_dim, void* out_host, float* lse_host,
                             float softmax_scale, void* q_dev, void* k_dev, void* v_dev,
                             int32_t* cu_seqlens_dev, void* worklist_dev, size_t worklist_bytes,
                             void* out_dev, float* lse_dev, void* stream);

/* Size in bytes of the static worklist array used by pva_attn_fwd_noalloc. */
size_t pva_noalloc_scratch_bytes(void);

/* Device error word of the last pva_attn_fwd_noalloc call on the current
 * device (0 = none; otherwise as pva_worklist_error: 100 capacity, 102 a
 * worklist that does not match, 200 + a wait site).  Synchronizes `stream`
 * (the stream of that call) and copies 4 bytes to code_out (HOST).  The pages
 * have no counterpart.  Allocates nothing. */
pva_status pva_noalloc_error(int32_t* code_out, void* stream);

/* Test hook for the failure path of the bounded waits (the pages have no
 * counterpart).  While `enable` is non-zero, pva_attn_fwd launches made by
 * this process tell one CTA's TMA producer (CTA 0's under STATIC dispatch,
 * that of the CTA which claimed the first unit under DYNAMIC) to skip its
 * second K/V load.  The
 * MMA warps of that CTA then wait for a copy that never comes; their bounded
 * wait (2 s) expires, the CTA raises its abort flag, drains its own copies and
 * MMAs, frees tensor memory and returns, and pva_worklist_error() reports
 * 200 + the wait site.  Nothing faults and the CUDA context stays usable;
 * every other CTA finishes its work.  For tests only. */
void pva_debug_withhold_kv_load(int32_t enable);

const char* pva_status_string(pva_status status);
int32_t pva_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PVA_H */
