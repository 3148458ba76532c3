/*
 * oracle.h -- declarations of the fp64 CPU oracle (test infrastructure only).
 * This header belongs to the oracle alone; the CUDA library never includes it.
 */
#ifndef PVA_ORACLE_H
#define PVA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Mask kinds (integer values agreed with the library's public header). */
enum {
    OR_MASK_CAUSAL = 0,
    OR_MASK_SLIDING_WINDOW = 1,
    OR_MASK_SHARED_QUESTION = 2,
    OR_MASK_ZIGZAG_PAIR = 3,
    OR_MASK_SLICES = 4,
    OR_MASK_ZIGZAG_STEP = 5
};
enum { OR_SLICE_FULL = 0, OR_SLICE_CAUSAL = 1, OR_SLICE_INV_CAUSAL = 2, OR_SLICE_BI_CAUSAL = 3,
       OR_SLICE_PACKED = 4 /* short documents sharing one tile (worklist only) */ };

typedef struct {
    int32_t kind;
    int32_t window;     /* sliding window: keys with q_pos - k_pos < window */
    int32_t num_prefix; /* shared question: documents [0, num_prefix) are questions */
    int32_t cp, q_rank, k_rank; /* zigzag pair */
    const int32_t *slices;      /* [num_slices][8]: q_row0 q_len q_pos0 k_row0 k_len k_pos0 type window */
    int32_t num_slices;
    int32_t ring_step;          /* zigzag ring step (with cp): every rank at step ring_step */
} or_mask_t;

int32_t or_num_threads(void);
int32_t or_zigzag_map(const int32_t *cu, int32_t ndocs, int32_t cp, int32_t rank, int32_t *map,
                      int32_t *chunk_table);
int or_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, int32_t Tq, int32_t Tk,
                 int32_t Hq, int32_t Hkv, int32_t d, const int32_t *cu, int32_t ndocs,
                 const or_mask_t *m, double scale, const int32_t *jobs, int64_t njobs,
                 int32_t brute, double *out, double *lse);
int or_attention_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const uint16_t *dout, int32_t Tq, int32_t Tk, int32_t Hq, int32_t Hkv,
                     int32_t d, const int32_t *cu, int32_t ndocs, const or_mask_t *m,
                     double scale, double *dq, double *dk, double *dv);
int or_attention_bwd_jobs(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const uint16_t *dout, int32_t Tq, int32_t Tk, int32_t Hq, int32_t Hkv,
                          int32_t d, const int32_t *cu, int32_t ndocs, const or_mask_t *m,
                          double scale, const int32_t *qjobs, int64_t nq, const int32_t *kjobs,
                          int64_t nk, double *dq, double *dk, double *dv);
int64_t or_pair_count(int32_t Tq, int32_t Tk, const int32_t *cu, int32_t ndocs,
                      const or_mask_t *m, int32_t brute);
int or_allowed_matrix(int32_t Tq, int32_t Tk, const int32_t *cu, int32_t ndocs,
                      const or_mask_t *m, uint8_t *out);
void or_merge(const double *oa, const double *la, const double *ob, const double *lb, double *o,
              double *l, int64_t tokens, int32_t heads, int32_t d);
int or_lpt(const int64_t *cost, int64_t n, int32_t bins, int32_t *assign, int64_t *order,
           int64_t *loads);
int or_refine_move_swap(const int64_t *cost, int64_t n, int32_t bins, int32_t *assign,
                        int64_t *loads, int32_t max_iters);
int64_t or_fit_tile_cost(const int64_t *P, const int64_t *U, const double *t, int32_t nb,
                         double *coef);
int or_worklist(const int32_t *cu, int32_t ndocs, const or_mask_t *m, int32_t tile_m,
                int32_t tile_n, int32_t Hq, int32_t Hkv, int32_t num_ctas, int64_t c_tile,
                int32_t refine_iters, int32_t pack_docs,
                int64_t *counts, int32_t *slices_out, uint32_t *slice_masks_out,
                int32_t *segs_out, int32_t *units_out,
                int64_t *unit_cost_out, int64_t *unit_pairs_out, int32_t *runs_out,
                int32_t *cta_off_out);

int or_chunk_areas(int32_t T, const int32_t *cu, int32_t ndocs, const or_mask_t *m,
                   int32_t chunk_size, int64_t *areas);
int or_dispatch_minheap(const int64_t *areas, int32_t n, int32_t cp, int32_t *bucket,
                        int64_t *loads);
int32_t or_striped_map(int32_t T, int32_t cp, int32_t rank, int32_t stripe, int32_t *map);
int or_wlb_choose(const int32_t *cu, int32_t ndocs, int32_t cp, int32_t tile, int32_t d,
                  int64_t *costs);

#ifdef __cplusplus
}
#endif
#endif
