// sched.cu - tile enumeration and ordering for the BDLM kernels.
//
// One small kernel, launched before every attention kernel, that
//   1. clears the workspace header (error word, work counter);
//   2. validates cu_seqlens / the block list on the device (a task list is
//      checked on the host and reaches the device through task_upload_kernel);
//   3. enumerates the row tiles of the call (never straddling a document half)
//      with a cost estimate in key tiles (forward) or query rows (backward);
//   4. orders them by descending cost with a counting sort (for a task list,
//      earlier tasks first among tiles of equal cost).
// The attention kernels then take work items from the front of this list with
// an atomic counter. Taking the heaviest remaining tile first is the
// work-conserving form of pairing early and late blocks for balance (rit.work
// CSBP post: the valid pairs are unchanged and early and late blocks are
// assigned together): the last blocks of a sequence carry the longest clean
// prefixes and are dealt first, the first blocks fill in behind them.
#include "common.cuh"
#include "kernels.h"

namespace bdlm {

namespace {

constexpr int kThreads = 1024;
constexpr int kBuckets = 8192;
constexpr int kTaskGroups = 64;  // task-order levels among tiles of equal cost

__device__ int block_exclusive_scan(int x, int* total, int* sbuf) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int v = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    if (lane == 31) sbuf[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = sbuf[lane];
        int ws = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, ws, o);
            if (lane >= o) ws += y;
        }
        sbuf[32 + lane] = ws - w;
        if (lane == 31) sbuf[64] = ws;
    }
    __syncthreads();
    int res = v - x + sbuf[32 + warp];
    *total = sbuf[64];
    __syncthreads();
    return res;
}

__device__ void doc_of(const Layout& lay, int d, int* start, int* n) {
    if (lay.mode == MODE_FULL && lay.cu) {
        int s = __ldg(lay.cu + d), e = __ldg(lay.cu + d + 1);
        *start = s;
        *n = (e - s) / 2;
    } else {
        *start = 0;
        *n = lay.n;
    }
}

// Cost of a forward query tile, in key tiles of kn rows.
__device__ int fwd_cost(const TileRange& g, int kn) {
    return (g.r1_hi - g.r1_lo + kn - 1) / kn + (g.r2_hi - g.r2_lo + kn - 1) / kn;
}

// Tiles of `rows` rows covering positions [lo, hi).
__device__ __forceinline__ int run_tiles(int lo, int hi, int rows) { return hi > lo ? (hi - lo + rows - 1) / rows : 0; }

// Cost of a backward key tile, in query rows that see it.
__device__ int bwd_cost(const Layout& lay, const Tile& t) {
    const KeyRows r = key_tile_rows(lay, t);
    return (r.a_hi - r.a_lo) + (r.b_hi - r.b_lo);
}

__global__ void __launch_bounds__(kThreads, 1)
enumerate_kernel(Layout lay, int tile_rows, int key_tile, int kind, Tile* table, Tile* tmp,
                 int* cost_tmp, TileRange* ranges, TileRange* rng_tmp, WsHeader* hdr, int max_tiles,
                 int cost_shift, int task_groups) {
    __shared__ int hist[kBuckets];
    __shared__ int sbuf[96];
    __shared__ int s_carry;
    __shared__ int s_off[kThreads];
    const int tid = threadIdx.x;
    if (tid == 0) {
        hdr->error = 0;
        hdr->info = 0;
        hdr->n_tiles = 0;
        hdr->counter = 0;
        s_carry = 0;
    }
    for (int i = tid; i < kBuckets; i += kThreads) hist[i] = 0;

    // ---- device-side validation -------------------------------------------
    int bad = 0, bad_info = 0;
    const int ndocs = (lay.mode == MODE_FULL && lay.cu) ? lay.n_docs : 1;
    if (lay.mode == MODE_FULL && lay.cu) {
        for (int d = tid; d < ndocs; d += kThreads) {
            long long s = __ldg(lay.cu + d), e = __ldg(lay.cu + d + 1);
            long long len = e - s;
            if (len <= 0 || (len & 1)) { bad = 1; bad_info = d; }  // [clean | corrupted] halves
        }
        if (tid == 0 && (__ldg(lay.cu) != 0 || (long long)__ldg(lay.cu + ndocs) != lay.L)) {
            bad = 1;
            bad_info = -1;
        }
    }
    if (lay.mode == MODE_GROUP) {
        const int nb = (lay.n + lay.B - 1) / lay.B;  // a short last block counts
        for (int i = tid; i < lay.n_blocks; i += kThreads) {
            int b = __ldg(lay.blocks + i);
            if (b < 0 || b >= nb) { bad = 1; bad_info = i; }
            // the key-major backward needs the list strictly ascending
            if (kind == 1 && i > 0 && b <= __ldg(lay.blocks + i - 1)) { bad = 1; bad_info = i; }
        }
    }
    if (__syncthreads_or(bad)) {
        if (bad) set_error(hdr, DEV_CHECK, bad_info);
        return;
    }

    // ---- enumeration ---------------------------------------------------------
    if (lay.mode == MODE_WINDOW || (kind == 1 && lay.mode == MODE_GROUP)) {
        // tiles in two runs that never straddle the clean/corrupted boundary:
        // forward - the window's query positions; backward - the window's key
        // positions, or the group's k rows (clean [0, n), then its corrupted rows)
        int c_lo, c_hi, x_lo, x_hi;
        if (lay.mode == MODE_WINDOW) {
            const int lo = kind == 0 ? lay.q_lo : lay.kw_lo, hi = kind == 0 ? lay.q_hi : lay.kw_hi;
            c_lo = lo;
            c_hi = imin(hi, lay.n);
            x_lo = imax(lo, lay.n);
            x_hi = hi;
        } else {
            c_lo = 0;
            c_hi = lay.n;
            x_lo = lay.n;
            x_hi = lay.n + lay.n_blocks * lay.B;
        }
        const int nc = c_hi > c_lo ? (c_hi - c_lo + tile_rows - 1) / tile_rows : 0;
        const int nx = x_hi > x_lo ? (x_hi - x_lo + tile_rows - 1) / tile_rows : 0;
        for (int i = tid; i < nc + nx && i < max_tiles; i += kThreads) {
            const bool cl = i < nc;
            const int p0 = cl ? c_lo + i * tile_rows : x_lo + (i - nc) * tile_rows;
            tmp[i] = Tile{0, lay.n, p0, imin(tile_rows, (cl ? c_hi : x_hi) - p0)};
        }
        if (tid == 0) s_carry = nc + nx;
        __syncthreads();
    } else if (lay.mode == MODE_TASKS) {
        // tasks in chunks of kThreads: scan the per-task tile counts (each
        // task's query positions (forward) or key positions (backward) in two
        // runs split at its clean/corrupted boundary), then let every thread
        // fill tiles, finding its task by binary search over the chunk's tile
        // offsets
        for (int base = 0; base < lay.n_tasks; base += kThreads) {
            const int ti = base + tid;
            const int nt = imin(kThreads, lay.n_tasks - base);
            int cnt = 0;
            if (ti < lay.n_tasks) {
                const TaskRec r = lay.tasks[ti];
                const int lo = kind == 0 ? r.q_lo : r.kw_lo, hi = kind == 0 ? r.q_hi : r.kw_hi;
                cnt = run_tiles(lo, imin(hi, r.n), tile_rows) + run_tiles(imax(lo, r.n), hi, tile_rows);
            }
            int total;
            const int off = block_exclusive_scan(cnt, &total, sbuf);
            s_off[tid] = off;
            __syncthreads();
            const int carry = s_carry;
            for (int i = tid; i < total; i += kThreads) {
                int lo = 0, hi = nt - 1;  // last task whose offset <= i
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s_off[mid] <= i) lo = mid; else hi = mid - 1;
                }
                const TaskRec r = lay.tasks[base + lo];
                const int a0 = kind == 0 ? r.q_lo : r.kw_lo, a1 = kind == 0 ? r.q_hi : r.kw_hi;
                const int li = i - s_off[lo];
                const int c_hi = imin(a1, r.n);
                const int nc = run_tiles(a0, c_hi, tile_rows);
                const int p0 = li < nc ? a0 + li * tile_rows : imax(a0, r.n) + (li - nc) * tile_rows;
                const int end = li < nc ? c_hi : a1;
                const int idx = carry + i;
                if (idx < max_tiles) tmp[idx] = Tile{r.seq_start, r.n, p0, imin(tile_rows, end - p0), base + lo};
            }
            __syncthreads();
            if (tid == 0) s_carry = carry + total;
            __syncthreads();
        }
    } else if (lay.mode == MODE_GROUP) {
        const int rows = lay.n_blocks * lay.B;
        const int nt = (rows + tile_rows - 1) / tile_rows;
        for (int i = tid; i < nt && i < max_tiles; i += kThreads)
            tmp[i] = Tile{0, lay.n, i * tile_rows, imin(tile_rows, rows - i * tile_rows)};
        if (tid == 0) s_carry = nt;
        __syncthreads();
    } else {
        // documents in chunks of kThreads: scan the per-document tile counts,
        // then let every thread fill tiles, finding its document by binary
        // search over the chunk's tile offsets
        for (int base = 0; base < ndocs; base += kThreads) {
            const int d = base + tid;
            const int nd = imin(kThreads, ndocs - base);
            int start = 0, n = 0, per_half = 0;
            if (d < ndocs) {
                doc_of(lay, d, &start, &n);
                per_half = (n + tile_rows - 1) / tile_rows;
            }
            int total;
            const int off = block_exclusive_scan(2 * per_half, &total, sbuf);
            s_off[tid] = off;
            __syncthreads();
            const int carry = s_carry;
            for (int i = tid; i < total; i += kThreads) {
                int lo = 0, hi = nd - 1;  // last document whose offset <= i
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s_off[mid] <= i) lo = mid; else hi = mid - 1;
                }
                int ds, dn;
                doc_of(lay, base + lo, &ds, &dn);
                const int ph = (dn + tile_rows - 1) / tile_rows;
                const int li = i - s_off[lo];
                const int half = li / ph, j = li % ph;
                const int p0 = half * dn + j * tile_rows;
                const int idx = carry + i;
                if (idx < max_tiles) tmp[idx] = Tile{ds, dn, p0, imin(tile_rows, (half + 1) * dn - p0)};
            }
            __syncthreads();
            if (tid == 0) s_carry = carry + total;
            __syncthreads();
        }
    }
    const int n_tiles = s_carry;
    if (n_tiles > max_tiles) {
        if (tid == 0) set_error(hdr, DEV_CHECK, -2);
        return;
    }
    __syncthreads();

    // ---- exact ranges and costs -------------------------------------------------
    for (int i = tid; i < n_tiles; i += kThreads) {
        const Tile t = tmp[i];
        int c;
        if (kind == 0) {
            const TileRange g = tile_range(lay, t);
            rng_tmp[i] = g;
            c = fwd_cost(g, key_tile);
        } else {
            c = bwd_cost(lay, t);
        }
        c = c >> cost_shift;
        // task lists: among tiles of equal cost, earlier tasks first, so
        // that the CTAs running side by side mostly share one task's keys
        if (task_groups > 1) c = c * task_groups + (task_groups - 1 - (int)((long long)t.task * task_groups / lay.n_tasks));
        c = imin(c, kBuckets - 1);
        cost_tmp[i] = c;
        atomicAdd(&hist[c], 1);
    }
    __syncthreads();

    // ---- counting sort, heaviest first ----------------------------------------
    // bucket c starts after all buckets c' > c
    constexpr int per = kBuckets / kThreads;
    const int first = kBuckets - (tid + 1) * per;  // thread 0 owns the top buckets
    int local = 0;
    for (int i = 0; i < per; ++i) local += hist[first + i];
    int total;
    int off = block_exclusive_scan(local, &total, sbuf);
    __syncthreads();
    {
        int run = off;
        for (int i = per - 1; i >= 0; --i) {
            int c = hist[first + i];
            hist[first + i] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int i = tid; i < n_tiles; i += kThreads) {
        int pos = atomicAdd(&hist[cost_tmp[i]], 1);
        table[pos] = tmp[i];
        if (kind == 0) ranges[pos] = rng_tmp[i];
    }
    if (tid == 0) hdr->n_tiles = n_tiles;
}

// Task records reach the device as kernel parameters (no host-to-device
// copy, and a captured launch keeps them by value).
struct TaskChunk {
    int count;
    int pad[7];
    TaskRec rec[kTaskUploadChunk];
};

__global__ void task_upload_kernel(const __grid_constant__ TaskChunk c, TaskRec* dst) {
    for (int i = threadIdx.x; i < c.count; i += blockDim.x) dst[i] = c.rec[i];
}

}  // namespace

int launch_task_upload(const TaskRec* host, int n, TaskRec* dst, cudaStream_t st) {
    int launches = 0;
    for (int base = 0; base < n; base += kTaskUploadChunk) {
        TaskChunk c;
        c.count = imin(kTaskUploadChunk, n - base);
        for (int i = 0; i < 7; ++i) c.pad[i] = 0;
        for (int i = 0; i < c.count; ++i) c.rec[i] = host[base + i];
        task_upload_kernel<<<1, 256, 0, st>>>(c, dst + base);
        ++launches;
    }
    return launches;
}

void launch_enumerate(const Layout& lay, int tile_rows, int key_tile, int kind, const WsCarve& ws,
                      cudaStream_t st) {
    // keep the costs inside the histogram for very long sequences (a task
    // list's lay.n is its longest sequence), with room for the task order
    const int groups = lay.mode == MODE_TASKS ? imin(lay.n_tasks, kTaskGroups) : 1;
    int shift = 0;
    long long max_cost = kind == 0 ? (2 * (long long)(lay.mode == MODE_FULL && lay.cu ? lay.L : lay.n)) / key_tile + 4
                                   : 2 * (long long)(lay.mode == MODE_FULL && lay.cu ? lay.L : lay.n);
    while (((max_cost >> shift) + 1) * groups > kBuckets) ++shift;
    enumerate_kernel<<<1, kThreads, 0, st>>>(lay, tile_rows, key_tile, kind, ws.table, ws.tmp, ws.cost,
                                             ws.ranges, ws.rng_tmp, ws.hdr, ws.max_tiles, shift, groups);
}

}  // namespace bdlm
