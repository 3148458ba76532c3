// wl_layout.cuh -- byte layout of the device worklist buffer.
//
// The buffer is owned by the caller; the host computes capacities and
// section offsets from bounds (pva_worklist_bytes), the device kernels fill
// it.  Sections (each 256-byte aligned):
//   header     WlHeader
//   slices     WlSlice[cap_slices]        slices of the mask, enumeration order
//   segs       WlSeg[cap_segs]            query segments (slices sharing a q range)
//   units_enum WlUnit[cap_units]          work units in enumeration order
//   keys       uint64[cap_units]          sort keys: (~cost << 24) | uid, then (cta << 24) | uid
//   order      int32[cap_units]           uid of the r-th unit in LPT order
//   assign     int32[cap_units]           bin (CTA) of each uid
//   units      WlUnit[cap_units]          units grouped by CTA, in enumeration order inside a CTA
//   runs       WlRun[cap_runs]            per unit and slice: kv tile span [lo, hi)
//   cta_off    int32[num_ctas + 1]        CSR offsets of the CTAs into `units`
//   doc_scan   int32[6 * (items + 1)]     per-document (or per rank and document) scan scratch
//   dorder     int32[cap_units]           uid of the r-th unit in dispatch order
//   cls_work   uint64[64]                 summed cost per dispatch class
//   smask      uint32[cap_slices][4]      per packed slice: rows that start a document
// A worklist built for dynamic dispatch has no LPT bins: order, assign,
// units and cta_off are left unwritten (units_enum and dorder describe it).
#pragma once

#include <stdint.h>

namespace pva {

constexpr int32_t kWlMagic = 0x57415650;  // "PVAW"
constexpr int32_t kWlVersion = 3;
constexpr int kMaxBins = 1024;
constexpr int kUidBits = 24;   // units per worklist < 2^24
constexpr int kCostBits = 40;  // unit cost < 2^40

struct WlSlice {
    int32_t q_row0, q_len, q_pos0, k_row0, k_len, k_pos0, type, window;
};

// Slice type of a tile shared by several short documents (built by the
// worklist, never passed in by a caller): a group of consecutive documents,
// each shorter than a tile, whose rows fit in one tile.  Its q and k ranges
// are the group's rows, positions count from the group's first row, and a
// row sees the keys of its own document at positions <= its own (and inside
// the window, if any).  Bit r of the slice's 128-bit smask entry is set when
// row r starts a document.
constexpr int32_t kSlicePacked = 4;

// First row of the document holding row r (0 <= r < 128) of a packed slice.
__host__ __device__ inline int32_t packed_doc_start(const uint32_t* m, int32_t r) {
    for (int32_t w = r >> 5; w >= 0; --w) {
        uint32_t bits = m[w];
        if (w == (r >> 5)) bits &= (r & 31) == 31 ? 0xffffffffu : ((2u << (r & 31)) - 1u);
        if (bits) {
#ifdef __CUDA_ARCH__
            return w * 32 + 31 - __clz(bits);
#else
            int32_t b = 31;
            while (!(bits >> b)) --b;
            return w * 32 + b;
#endif
        }
    }
    return 0;
}

// One past the last row of the document holding row r of a packed slice of
// `len` rows.
__host__ __device__ inline int32_t packed_doc_end(const uint32_t* m, int32_t r, int32_t len) {
    for (int32_t w = (r + 1) >> 5; w < 4 && w * 32 < len; ++w) {
        uint32_t bits = m[w];
        if (w == ((r + 1) >> 5)) bits &= ~((1u << ((r + 1) & 31)) - 1u);
        if (bits) {
#ifdef __CUDA_ARCH__
            const int32_t b = w * 32 + __ffs(bits) - 1;
#else
            int32_t z = 0;
            while (!((bits >> z) & 1u)) ++z;
            const int32_t b = w * 32 + z;
#endif
            return b < len ? b : len;
        }
    }
    return len;
}

struct WlSeg {
    int32_t q_row0, q_len, q_pos0, slice_begin, slice_count, unit_base, run_base, ntiles;
};

struct WlUnit {
    int32_t uid, seg, t0, t1, h0, h1, kvh, run_begin, run_count, cta, ntiles, pad;
    int64_t cost, pairs;
};
static_assert(sizeof(WlUnit) == 64, "WlUnit is 64 bytes");

// Dispatch class of a unit: floor(log2(max(cost, 1))).  The dynamic dispatch
// order: classes above a split class in decreasing order, units of one class
// in enumeration order (segment, kv head, head pair, q tile), so that CTAs
// running at the same time share the same documents' K/V in L2; then every
// unit of the split class and below in exact LPT order (cost desc, uid asc).
// The split is the highest class c whose units could not be absorbed by the
// work below it: W(classes < c) < num_ctas * 2^(c + 1) (capped at 38, so that
// the LPT part's costs fit the sort key).
__host__ __device__ inline int32_t dispatch_class(int64_t cost) {
    const uint64_t c = cost > 1 ? (uint64_t)cost : 1u;
#ifdef __CUDA_ARCH__
    return 63 - __clzll((long long)c);
#else
    int32_t e = 0;
    for (uint64_t x = c; x >>= 1;) ++e;
    return e;
#endif
}

struct WlRun {
    int32_t slice, lo, hi, pad;
};

struct WlOffsets {
    int64_t slices, segs, units_enum, keys, order, assign, units, runs, cta_off, doc_scan, dorder,
        cls_work, smask, total;
};

struct WlHeader {
    int32_t magic, version;
    int32_t error;     // device error word (0 = none)
    int32_t num_ctas;
    int32_t tile_m, tile_n, hq, hkv;
    int32_t kind, q_tokens, k_tokens, num_docs;
    int32_t cap_slices, cap_segs, cap_units, cap_runs;
    int32_t nslices, nsegs, nunits, nruns;  // written by the device
    int64_t c_tile;
    unsigned long long pair_sum;   // sum over units of allowed pairs (all sub-tiles)
    unsigned long long tile_sum;   // sum over units of sub-tiles x kv tiles
    WlOffsets off;
    int32_t lpt_steps;  // batches + runs taken by the LPT (diagnostic)
    int32_t refine_iters;   // move/swap rounds allowed after LPT
    int32_t refine_rounds;  // move/swap rounds applied (diagnostic)
    // Dynamic dispatch of the forward kernel: the next rank of `dorder` to hand
    // out and the CTAs that have finished; the last CTA to finish puts both
    // back to 0.
    int32_t dispatch_next, dispatch_done;
    int32_t dispatch;  // pva_dispatch the worklist was built for (dorder exists if DYNAMIC)
    int32_t dispatch_split;  // classes <= this one are dispatched in exact LPT order
    int32_t pack_docs;       // short documents share tiles (pva_worklist_params.pack_docs)
};
static_assert(sizeof(WlHeader) <= 256, "header fits in 256 bytes");

// Backward plan: kv-major units.  Slices with the same key range form a key
// group (a document's keys under a causal mask; a question's keys shared by
// its own slice and every answer's; a zigzag key chunk seen by two query
// chunks); different groups' key ranges are disjoint.  A unit is one 128-key
// tile of a group for one kv head; it covers every slice of the group and
// every head of the kv head's group, so each key row has one writer.
// Buffer sections (256-byte aligned): header, units, sort keys, order (rank ->
// unit), gslices (slice indices sorted by key range), D scratch [hq, q_tokens].
constexpr int32_t kBwdMagic = 0x42415650;  // "PVAB"
constexpr int32_t kBwdMaxSlices = 8192;    // slices the plan kernel groups in shared memory

struct BwdUnit {
    int32_t gbegin, gcount;  // the group's slices: gslices[gbegin, gbegin + gcount)
    int32_t kt, kvh;
    int64_t cost;  // q-tile steps over the group's slices and heads + 1
};
static_assert(sizeof(BwdUnit) == 24, "BwdUnit is 24 bytes");

struct BwdHeader {
    int32_t magic, error, nunits, cap_units;
    int32_t hq, hkv, q_tokens, k_tokens;
    int32_t dispatch_next, dispatch_done;  // dynamic dispatch counter of the dK/dV pass
    int64_t off_units, off_keys, off_order, off_gslices, off_dvec, total;
};
static_assert(sizeof(BwdHeader) <= 256, "backward header fits in 256 bytes");

// The slice MaskTypes (pva_slice_type), on token positions: CAUSAL k <= q,
// INV_CAUSAL k >= q (each with an optional window |q - k| < w), BI_CAUSAL
// k >= q and k_end - k >= q_end - q.
// Keys of slice s a query at position qp may see, as slice-local key indices
// [lo, hi) (empty when hi <= lo).  pm: the slice's smask entry (packed slices).
__host__ __device__ inline void slice_keys_of_query(const WlSlice& s, int64_t qp, int64_t& lo,
                                                    int64_t& hi, const uint32_t* pm = nullptr) {
    const int64_t d = qp - s.k_pos0;  // local index of the key at the query's position
    lo = 0;
    hi = s.k_len;
    if (s.type == kSlicePacked) {  // own document, causal (positions = rows of the group)
        const int32_t r = (int32_t)(qp - s.q_pos0);
        lo = pm ? packed_doc_start(pm, r) : r;
        hi = d + 1;
        if (s.window > 0 && d - s.window + 1 > lo) lo = d - s.window + 1;
    } else if (s.type == 1) {  // CAUSAL
        hi = d + 1;
        if (s.window > 0) lo = d - s.window + 1;
    } else if (s.type == 2) {  // INV_CAUSAL
        lo = d;
        if (s.window > 0) hi = d + s.window;
    } else if (s.type == 3) {  // BI_CAUSAL: local key j <= k_len - q_len + local row
        lo = d;
        hi = (int64_t)s.k_len - s.q_len + (qp - s.q_pos0) + 1;
    }
    if (lo < 0) lo = 0;
    if (hi > s.k_len) hi = s.k_len;
}

// Query positions [lo, hi) of slice s that may see a key at position kp (both
// ends are non-decreasing in kp for every type).
__host__ __device__ inline void slice_queries_of_key(const WlSlice& s, int64_t kp, int64_t& lo,
                                                     int64_t& hi, const uint32_t* pm = nullptr) {
    lo = s.q_pos0;
    hi = (int64_t)s.q_pos0 + s.q_len;
    int64_t a = lo, b = hi;
    if (s.type == kSlicePacked) {  // the key's document, from the key's position on
        const int32_t j = (int32_t)(kp - s.k_pos0);
        a = kp;
        b = (int64_t)s.q_pos0 + (pm ? packed_doc_end(pm, j, s.q_len) : j + 1);
        if (s.window > 0 && kp + s.window < b) b = kp + s.window;
    } else if (s.type == 1) {  // CAUSAL
        a = kp;
        if (s.window > 0) b = kp + s.window;
    } else if (s.type == 2) {  // INV_CAUSAL
        b = kp + 1;
        if (s.window > 0) a = kp - s.window + 1;
    } else if (s.type == 3) {  // BI_CAUSAL: q >= q_end - k_end + k
        b = kp + 1;
        a = ((int64_t)s.q_pos0 + s.q_len) - ((int64_t)s.k_pos0 + s.k_len) + kp;
    }
    if (a > lo) lo = a;
    if (b < hi) hi = b;
}

// q tiles [qlo, qhi) of slice `sl` (aligned at its query start, like the
// forward) holding a row that may see a key of key tile kt of the slice.
__host__ __device__ inline void bwd_q_span(const WlSlice& sl, int32_t kt, int32_t& qlo,
                                           int32_t& qhi, const uint32_t* pm = nullptr) {
    const int32_t ka = kt * 128, kb = (sl.k_len < ka + 128) ? sl.k_len : ka + 128;
    qlo = qhi = 0;
    if (kb <= ka) return;
    int64_t a0, a1, b0, b1;
    slice_queries_of_key(sl, (int64_t)sl.k_pos0 + ka, a0, a1, pm);
    slice_queries_of_key(sl, (int64_t)sl.k_pos0 + kb - 1, b0, b1, pm);
    const int64_t r_lo = a0 - sl.q_pos0, r_hi = b1 - sl.q_pos0;
    if (r_hi <= r_lo) return;
    qlo = (int32_t)(r_lo / 128);
    qhi = (int32_t)((r_hi + 127) / 128);
}

// The smask entry of slice `si` if it is a packed slice, else nullptr.
__host__ __device__ inline const uint32_t* slice_mask(const uint8_t* wl, const WlHeader* h,
                                                      const WlSlice& s, int32_t si) {
    return s.type == kSlicePacked
               ? reinterpret_cast<const uint32_t*>(wl + h->off.smask) + 4 * (int64_t)si
               : nullptr;
}

// Device error codes (stored in WlHeader::error).
enum : int32_t {
    kErrNone = 0,
    kErrCapacity = 100,       // a count exceeded its capacity
    kErrCostRange = 101,      // a unit cost does not fit the sort key
    kErrBadWorklist = 102,    // attention called with a worklist that does not match
    kErrTimeoutBase = 200     // + wait site id: a bounded wait expired
};

}  // namespace pva
