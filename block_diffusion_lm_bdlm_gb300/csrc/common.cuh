// common.cuh - layout decode shared by the BDLM kernels.
//
// Blocks are cut from the start of each half of a document; when B does not
// divide the half's length n, the last block holds n mod B rows. Every query
// row of a call has at most two key intervals, in k-row coordinates of the
// call's k/v buffers:
//   prefix [p_lo, p_hi): the clean keys it sees (clean blocks <= b for a clean
//                        row of block b, clean blocks < b for a corrupted row),
//   diag   [d_lo, d_hi): its own corrupted block (corrupted rows only).
// This is the BDLM mask of "Block Parallelism For Efficient Distributed
// Long-Context Diffusion Language Model Training" (abstract) and the rit.work
// CSBP post (first section), restated per row so that a tile of rows iterates
// contiguous key ranges and only boundary tiles need an element mask.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bdlm {

enum Mode : int { MODE_FULL = 0, MODE_WINDOW = 1, MODE_GROUP = 2, MODE_TASKS = 3 };

// Status codes written to the device error word (same values as bdlm.h).
enum DevStatus : int { DEV_OK = 0, DEV_TIMEOUT = 5, DEV_CHECK = 6 };

// First 256 bytes of every workspace.
struct WsHeader {
    int error;     // first device error (0 = none)
    int info;      // detail of the first error (e.g. offending document)
    int n_tiles;   // tiles enumerated by the prologue
    int counter;   // dynamic work counter of the main kernel
    int pad[60];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// One token-level task of a task-list forward, as the kernels read it: the
// query positions [q_lo, q_hi) of the sequence at rows [seq_start,
// seq_start + 2n) of q, k, v against its key positions [kw_lo, kw_hi);
// results go to output slot `slot`.
struct TaskRec {
    int seq_start, n;
    int kw_lo, kw_hi;
    int q_lo, q_hi;
    int slot, pad;
};
static_assert(sizeof(TaskRec) == 32, "task record is 32 bytes");

// How the rows of a call map to sequence positions.
struct Layout {
    int mode;
    int B;             // diffusion block size
    int n;             // clean length (single sequence / window / group)
    int kw_lo, kw_hi;  // MODE_WINDOW: key positions held by k/v
    int q_lo, q_hi;    // MODE_WINDOW: query positions held by q (q row = position - q_lo)
    const int* cu;     // MODE_FULL: device cu_seqlens, or nullptr for one sequence
    int n_docs;
    long long L;       // rows of the full concatenation
    const int* blocks; // MODE_GROUP: device list of corrupted block ids
    int n_blocks;
    const TaskRec* tasks;  // MODE_TASKS: device task records
    int n_tasks;
};

// One tile of consecutive rows that never straddles a document half.
// q row of tile row r = doc_start + pos0 + r.
struct Tile {
    int doc_start;  // first row of the document (0 for window / group)
    int n;          // clean length of the document
    int pos0;       // document position (full/window/tasks) or list row (group) of row 0
    int nrows;      // valid rows (<= tile height)
    int task;       // MODE_TASKS: index of the tile's task
};

struct Span {
    int p_lo, p_hi, d_lo, d_hi;
};

// Key ranges of a whole tile, in k rows: every row's prefix interval lies in
// [r1_lo, r1_hi) and every own-block interval in [r2_lo, r2_hi) (empty ranges
// are [0, 0)); a key window [k0, k0 + w) inside [full_lo, full_hi) is visible
// to every valid row of the tile, so it needs no element mask.
struct TileRange {
    int r1_lo, r1_hi, r2_lo, r2_hi;
    int full_lo, full_hi, pad0, pad1;
};

__host__ __device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int imax(int a, int b) { return a > b ? a : b; }

// Read-only load (through the read-only cache on the device). The layout
// helpers below also compile for the host, where the tests check them.
__host__ __device__ __forceinline__ int ld_ro(const int* p) {
#ifdef __CUDA_ARCH__
    return __ldg(p);
#else
    return *p;
#endif
}

// Rows of block b of a half of length n (the last block is short when B does
// not divide n). A block group gives every listed block B rows; the rows of
// a short block past the half's end are padding.
__host__ __device__ __forceinline__ int block_len(int n, int B, int b) { return imin(B, n - b * B); }

// Key intervals of tile row r (empty intervals are [0, 0)).
__host__ __device__ __forceinline__ Span row_span(const Layout& lay, const Tile& t, int r) {
    Span s{0, 0, 0, 0};
    if (r >= t.nrows) return s;
    const int B = lay.B;
    if (lay.mode == MODE_GROUP) {
        const int j = t.pos0 + r;
        const int li = j / B;
        const int b = ld_ro(lay.blocks + li);
        const int len = block_len(lay.n, B, b);
        if (j - li * B >= len) return s;  // padding row of a short last block
        if (b > 0) { s.p_lo = 0; s.p_hi = b * B; }
        s.d_lo = lay.n + li * B;
        s.d_hi = s.d_lo + len;
        return s;
    }
    const int n = t.n;
    const int pos = t.pos0 + r;
    // key window and k row of key position 0: a window's k/v hold only its
    // keys; a task's k/v hold every row, its window bounds the positions
    int kw_lo = 0, kw_hi = 2 * n, kbase = t.doc_start;
    if (lay.mode == MODE_WINDOW) {
        kw_lo = lay.kw_lo;
        kw_hi = lay.kw_hi;
        kbase -= kw_lo;
    } else if (lay.mode == MODE_TASKS) {
        kw_lo = ld_ro(&lay.tasks[t.task].kw_lo);
        kw_hi = ld_ro(&lay.tasks[t.task].kw_hi);
    }
    int pref_hi, dlo = 0, dhi = 0;
    if (pos < n) {
        pref_hi = (pos / B + 1) * B;
    } else {
        const int b = (pos - n) / B;
        pref_hi = b * B;
        dlo = n + b * B;
        dhi = dlo + B;
    }
    int lo = imax(0, kw_lo), hi = imin(pref_hi, imin(kw_hi, n));
    if (hi > lo) { s.p_lo = kbase + lo; s.p_hi = kbase + hi; }
    lo = imax(dlo, kw_lo);
    hi = imin(dhi, kw_hi);
    if (dhi > dlo && hi > lo) { s.d_lo = kbase + lo; s.d_hi = kbase + hi; }
    return s;
}

// Exact key ranges of tile t: one span per diffusion block of rows (all rows
// of a block share one span).
__host__ __device__ __forceinline__ TileRange tile_range(const Layout& lay, const Tile& t) {
    TileRange g{0x7fffffff, 0, 0x7fffffff, 0, 0, 0x7fffffff, 0, 0};
    const int B = lay.B;
    for (int r = 0; r < t.nrows;) {
        const Span s = row_span(lay, t, r);
        if (s.p_hi > s.p_lo) {
            g.r1_lo = imin(g.r1_lo, s.p_lo);
            g.r1_hi = imax(g.r1_hi, s.p_hi);
            g.full_lo = imax(g.full_lo, s.p_lo);
            g.full_hi = imin(g.full_hi, s.p_hi);
        } else {
            g.full_hi = 0;
        }
        if (s.d_hi > s.d_lo) {
            g.r2_lo = imin(g.r2_lo, s.d_lo);
            g.r2_hi = imax(g.r2_hi, s.d_hi);
        }
        if (lay.mode == MODE_GROUP) {  // padding rows of a short block in the tile see nothing
            const int li = (t.pos0 + r) / B;
            const int len = block_len(lay.n, B, ld_ro(lay.blocks + li));
            if (len < B && li * B + len < t.pos0 + t.nrows) g.full_hi = 0;
        }
        // first row of the next block; blocks are cut from the start of each
        // half (a group's list rows from 0), which is not a multiple of B when
        // B does not divide n
        const int pos = t.pos0 + r;
        const int half0 = (lay.mode == MODE_GROUP || pos < t.n) ? 0 : t.n;
        const int nxt = half0 + ((pos - half0) / B + 1) * B - t.pos0;
        r = nxt > r ? nxt : r + 1;
    }
    if (g.r1_hi == 0) g.r1_lo = 0;
    if (g.r2_hi == 0) g.r2_lo = 0;
    if (g.full_hi < g.full_lo) { g.full_lo = 0; g.full_hi = 0; }
    return g;
}

__host__ __device__ __forceinline__ bool span_sees(const Span& s, int kr) {
    return (kr >= s.p_lo && kr < s.p_hi) || (kr >= s.d_lo && kr < s.d_hi);
}

// The one interval a key tile of a forward range is masked with: the prefix
// interval while iterating the prefix range, the own-block interval while
// iterating the own-block range. (The last tile of the prefix range may run
// past the clean keys into own-block keys; those are counted by the own-block
// range only.) Returned as [lo, lo + len) relative to the tile's first key k0.
struct RelInterval {
    int lo;
    unsigned len;
};
__host__ __device__ __forceinline__ RelInterval range_interval(const Span& s, bool prefix, int k0) {
    const int lo = prefix ? s.p_lo : s.d_lo, hi = prefix ? s.p_hi : s.d_hi;
    return RelInterval{lo - k0, (unsigned)(hi > lo ? hi - lo : 0)};
}
__host__ __device__ __forceinline__ bool rel_sees(const RelInterval& r, int e) { return (unsigned)(e - r.lo) < r.len; }

// ---------------------------------------------------------------------------
// Key-major view (backward). A backward tile is a run of consecutive keys that
// never straddles the clean/corrupted boundary. Tile.pos0 is the sequence
// position of key 0 (full and tasks: document position; window: global
// position) or, for a block group, its k row (clean keys [0, n), then the
// group's corrupted rows). "Row positions" of the query side map to q rows as
// doc_start + p (full, tasks), p - q_lo (window) or the list row p (group).
// ---------------------------------------------------------------------------

// Number of list entries with block id <= b. The backward requires a strictly
// ascending block list, so the group rows that see a clean key of block b are
// the list rows from group_count_le(b) * B on.
__host__ __device__ __forceinline__ int group_count_le(const Layout& lay, int b) {
    int lo = 0, hi = lay.n_blocks;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (ld_ro(lay.blocks + mid) <= b) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// q row of row position p of a tile (full and tasks: sequence start +
// position; window: position - q_lo; group: the list row itself).
__host__ __device__ __forceinline__ int q_row_of(const Layout& lay, const Tile& t, int p) {
    return t.doc_start + p - (lay.mode == MODE_WINDOW ? lay.q_lo : 0);
}

// k row of key 0 of backward tile t.
__host__ __device__ __forceinline__ int key_row0(const Layout& lay, const Tile& t) {
    return lay.mode == MODE_WINDOW ? t.pos0 - lay.kw_lo : t.doc_start + t.pos0;
}

// The query rows that see key tile t: at most two row-position ranges (range
// a, then range b; empty ranges are [0, 0)). For a clean key of block b the
// rows are the clean rows of blocks >= b and the corrupted rows of blocks > b;
// for a corrupted key, the corrupted rows of its own block.
struct KeyRows {
    int a_lo, a_hi, b_lo, b_hi;
};
// Rows of a block group's list that hold real rows: all n_blocks * B, less
// the padding of the short last block when the (ascending) list ends with it.
__host__ __device__ __forceinline__ int group_rows_real(const Layout& lay) {
    const int B = lay.B, nbk = (lay.n + B - 1) / B;
    const int last = ld_ro(lay.blocks + lay.n_blocks - 1);
    return (lay.n_blocks - 1) * B + (last == nbk - 1 ? block_len(lay.n, B, last) : B);
}

__host__ __device__ __forceinline__ KeyRows key_tile_rows(const Layout& lay, const Tile& t) {
    KeyRows r{0, 0, 0, 0};
    const int n = t.n, B = lay.B;
    if (lay.mode == MODE_GROUP) {
        const int R = group_rows_real(lay);
        if (t.pos0 < n) {
            const int lo = group_count_le(lay, t.pos0 / B) * B;
            if (lo < R) { r.a_lo = lo; r.a_hi = R; }
        } else {
            r.a_lo = ((t.pos0 - n) / B) * B;
            r.a_hi = imin(((t.pos0 + t.nrows - 1 - n) / B + 1) * B, R);
            if (r.a_hi <= r.a_lo) { r.a_lo = 0; r.a_hi = 0; }  // padding keys only
        }
        return r;
    }
    if (t.pos0 < n) {
        const int b = t.pos0 / B;
        r.a_lo = b * B;
        r.a_hi = n;
        if ((b + 1) * B < n) { r.b_lo = n + (b + 1) * B; r.b_hi = 2 * n; }
    } else {
        r.a_lo = n + ((t.pos0 - n) / B) * B;
        r.a_hi = imin(n + ((t.pos0 + t.nrows - 1 - n) / B + 1) * B, 2 * n);  // a last block may be short
    }
    if (lay.mode == MODE_WINDOW || lay.mode == MODE_TASKS) {  // only the call's (task's) query rows
        const int qlo = lay.mode == MODE_WINDOW ? lay.q_lo : ld_ro(&lay.tasks[t.task].q_lo);
        const int qhi = lay.mode == MODE_WINDOW ? lay.q_hi : ld_ro(&lay.tasks[t.task].q_hi);
        r.a_lo = imax(r.a_lo, qlo);
        r.a_hi = imin(r.a_hi, qhi);
        if (r.a_hi <= r.a_lo) { r.a_lo = 0; r.a_hi = 0; }
        r.b_lo = imax(r.b_lo, qlo);
        r.b_hi = imin(r.b_hi, qhi);
        if (r.b_hi <= r.b_lo) { r.b_lo = 0; r.b_hi = 0; }
    }
    return r;
}

// The same for key kk of tile t alone (one interval per range; all empty for
// kk >= t.nrows).
__host__ __device__ __forceinline__ KeyRows key_rows(const Layout& lay, const Tile& t, int kk) {
    KeyRows r{0, 0, 0, 0};
    if (kk >= t.nrows) return r;
    const int n = t.n, B = lay.B, kc = t.pos0 + kk;
    if (lay.mode == MODE_GROUP) {
        if (kc < n) {
            r.a_lo = group_count_le(lay, kc / B) * B;
            r.a_hi = group_rows_real(lay);
            if (r.a_hi <= r.a_lo) { r.a_lo = 0; r.a_hi = 0; }
        } else {
            const int li = (kc - n) / B;
            const int len = block_len(n, B, ld_ro(lay.blocks + li));
            if (kc - n - li * B < len) {  // a real key: the real rows of its block
                r.a_lo = li * B;
                r.a_hi = r.a_lo + len;
            }
        }
        return r;
    }
    if (kc < n) {
        const int bk = kc / B;
        r.a_lo = bk * B;
        r.a_hi = n;
        r.b_lo = n + (bk + 1) * B;  // empty when the key's block is the last
        r.b_hi = 2 * n;
    } else {
        r.a_lo = n + ((kc - n) / B) * B;
        r.a_hi = imin(r.a_lo + B, 2 * n);  // a last block may be short
    }
    return r;
}

__device__ __forceinline__ void set_error(WsHeader* h, int code, int info) {
    if (atomicCAS(&h->error, 0, code) == 0) atomicExch(&h->info, info);
}

}  // namespace bdlm
