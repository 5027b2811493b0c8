// bdlm_api.cu - the C ABI declared in include/bdlm.h: host-side validation,
// workspace carving and kernel launches. No allocation, no synchronisation
// (except bdlm_read_error), no host<->device copies on the compute calls.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "bdlm.h"
#include "common.cuh"
#include "kernels.h"

using namespace bdlm;

namespace {

thread_local int g_launches = 0;

constexpr long long kMaxRows = 1LL << 30;  // row indices stay in int32

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int num_sms() {
    static int cache[128] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

long long max_tiles_for(long long L, int n_docs) {
    // the kernels enumerate tiles of 128 rows (keys); this bound allows one
    // per 64, with room to spare, plus one ragged tile per document half
    return L / 64 + 2LL * (n_docs > 0 ? n_docs : 1) + 4;
}

size_t sched_bytes_mt(long long mt) {
    size_t b = sizeof(WsHeader);
    b += round_up((size_t)mt * sizeof(Tile), 256);  // table
    b += round_up((size_t)mt * sizeof(Tile), 256);  // tmp
    b += round_up((size_t)mt * sizeof(int), 256);   // cost
    b += 2 * round_up((size_t)mt * sizeof(TileRange), 256);  // ranges, rng_tmp
    return b;
}

size_t sched_bytes(long long L, int n_docs) { return sched_bytes_mt(max_tiles_for(L, n_docs)); }

// Workspace carve-up for at most mt tiles; then, for the backward, D and the
// dq accumulator; then, for a task list, its n_tasks records.
WsCarve carve_mt(void* ws, long long mt, long long L, int H, int d, bool bwd, int n_tasks) {
    WsCarve c{};
    uint8_t* p = static_cast<uint8_t*>(ws);
    c.hdr = reinterpret_cast<WsHeader*>(p);
    p += sizeof(WsHeader);
    c.table = reinterpret_cast<Tile*>(p);
    p += round_up((size_t)mt * sizeof(Tile), 256);
    c.tmp = reinterpret_cast<Tile*>(p);
    p += round_up((size_t)mt * sizeof(Tile), 256);
    c.cost = reinterpret_cast<int*>(p);
    p += round_up((size_t)mt * sizeof(int), 256);
    c.ranges = reinterpret_cast<TileRange*>(p);
    p += round_up((size_t)mt * sizeof(TileRange), 256);
    c.rng_tmp = reinterpret_cast<TileRange*>(p);
    p += round_up((size_t)mt * sizeof(TileRange), 256);
    c.max_tiles = (int)mt;
    if (bwd) {
        c.D = reinterpret_cast<float*>(p);
        p += round_up((size_t)L * H * sizeof(float), 256);
        c.dqacc = reinterpret_cast<float*>(p);
        p += round_up((size_t)L * H * d * sizeof(float), 256);
    }
    if (n_tasks > 0) c.tasks = reinterpret_cast<TaskRec*>(p);
    return c;
}

WsCarve carve(void* ws, long long L, int n_docs, int H, int d, bool bwd) {
    return carve_mt(ws, max_tiles_for(L, n_docs), L, H, d, bwd, 0);
}

constexpr int kMaxTasks = 65536;
constexpr int kMaxSlots = 1024;

// Tiles of one task: forward - its query positions in 128-row tiles;
// backward - its key positions in 128-key tiles; each in two runs split at n.
long long task_tiles(const bdlm_task& t, bool bwd) {
    const long long rows = bwd ? kBwdKeyTile : kFwdTileRows;
    auto run = [rows](long long lo, long long hi) { return hi > lo ? (hi - lo + rows - 1) / rows : 0; };
    const long long lo = bwd ? t.key_lo : t.q_lo, hi = bwd ? t.key_hi : t.q_hi;
    const long long n = t.n;
    return run(lo, std::min(hi, n)) + run(std::max(lo, n), hi);
}

// Tile bound of a task list; -1 for an empty list or a task of empty size.
long long tasks_max_tiles(const bdlm_task* tasks, int n_tasks, bool bwd) {
    if (!tasks || n_tasks < 1 || n_tasks > kMaxTasks) return -1;
    long long mt = 4;
    for (int i = 0; i < n_tasks; ++i) {
        const bdlm_task& t = tasks[i];
        if (t.n <= 0 || t.n > kMaxRows || t.q_hi <= t.q_lo || t.q_hi - t.q_lo > kMaxRows) return -1;
        if (bwd && (t.key_hi <= t.key_lo || t.key_hi - t.key_lo > kMaxRows)) return -1;
        mt += task_tiles(t, bwd);
    }
    return mt;
}

// Host checks of a task list (every task inside its sequence, every sequence
// inside [0, L); the tasks of one slot write disjoint rows of q (forward) or
// of k (backward)); fills the device records and the longest clean length.
int check_tasks(const bdlm_task* tasks, int n_tasks, long long L, int n_slots, bool bwd, std::vector<TaskRec>* rec,
                long long* max_n) {
    if (!tasks || n_tasks < 1 || n_tasks > kMaxTasks || n_slots < 1 || n_slots > kMaxSlots) return BDLM_ERR_INVALID_ARG;
    rec->assign((size_t)n_tasks, TaskRec{});
    *max_n = 1;
    for (int i = 0; i < n_tasks; ++i) {
        const bdlm_task& t = tasks[i];
        if (t.reserved != 0 || t.slot < 0 || t.slot >= n_slots) return BDLM_ERR_INVALID_ARG;
        if (t.seq_start < 0 || t.n < 1 || t.n > L / 2 || t.seq_start > L - 2 * t.n) return BDLM_ERR_INVALID_ARG;
        if (t.q_lo < 0 || t.q_hi <= t.q_lo || t.q_hi > 2 * t.n) return BDLM_ERR_INVALID_ARG;
        if (t.key_lo < 0 || t.key_hi <= t.key_lo || t.key_hi > 2 * t.n) return BDLM_ERR_INVALID_ARG;
        (*rec)[i] = TaskRec{(int)t.seq_start, (int)t.n, (int)t.key_lo, (int)t.key_hi, (int)t.q_lo, (int)t.q_hi, t.slot, 0};
        *max_n = std::max(*max_n, (long long)t.n);
    }
    std::vector<int> ord((size_t)n_tasks);
    for (int i = 0; i < n_tasks; ++i) ord[i] = i;
    const std::vector<TaskRec>& r = *rec;
    auto lo = [&](int i) { return (long long)r[i].seq_start + (bwd ? r[i].kw_lo : r[i].q_lo); };
    auto hi = [&](int i) { return (long long)r[i].seq_start + (bwd ? r[i].kw_hi : r[i].q_hi); };
    std::sort(ord.begin(), ord.end(), [&](int a, int b) { return r[a].slot != r[b].slot ? r[a].slot < r[b].slot : lo(a) < lo(b); });
    for (int i = 1; i < n_tasks; ++i)
        if (r[ord[i - 1]].slot == r[ord[i]].slot && lo(ord[i]) < hi(ord[i - 1])) return BDLM_ERR_INVALID_ARG;
    return BDLM_OK;
}

struct Common {
    int mode;
    long long Lq, Lk;
    int n;
};

// Checks shared by fwd and bwd; fills Layout and the row counts.
int check_common(const void* q, const void* k, const void* v, long long L, int block, int heads,
                 int kv_heads, int head_dim, const int32_t* cu, int n_docs, const bdlm_partial* part,
                 Layout* lay, Common* cm) {
    if (!q || !k || !v) return BDLM_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return BDLM_ERR_INVALID_ARG;
    if (L <= 0 || L > kMaxRows || block <= 0 || heads <= 0 || kv_heads <= 0) return BDLM_ERR_INVALID_ARG;
    if (heads % kv_heads != 0) return BDLM_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return BDLM_ERR_UNSUPPORTED;
    const int kind = part ? part->kind : BDLM_PART_NONE;
    if (kind != BDLM_PART_NONE && kind != BDLM_PART_KEY_WINDOW && kind != BDLM_PART_BLOCK_GROUP)
        return BDLM_ERR_INVALID_ARG;
    std::memset(lay, 0, sizeof(*lay));
    lay->B = block;
    lay->L = L;
    if (cu) {
        if (kind != BDLM_PART_NONE) return BDLM_ERR_UNSUPPORTED;
        if (n_docs <= 0 || (long long)n_docs * 2 > L) return BDLM_ERR_INVALID_ARG;
        if (!aligned16(cu) && (reinterpret_cast<uintptr_t>(cu) & 3u)) return BDLM_ERR_INVALID_ARG;
        lay->mode = MODE_FULL;
        lay->cu = cu;
        lay->n_docs = n_docs;
        cm->mode = MODE_FULL;
        cm->Lq = cm->Lk = L;
        cm->n = 0;
        return BDLM_OK;
    }
    if (L % 2 != 0) return BDLM_ERR_INVALID_ARG;
    const long long n = L / 2;  // any n: a last block may be short
    lay->n = (int)n;
    lay->n_docs = 1;
    cm->n = (int)n;
    if (kind == BDLM_PART_NONE) {
        lay->mode = MODE_FULL;
        cm->mode = MODE_FULL;
        cm->Lq = cm->Lk = L;
    } else if (kind == BDLM_PART_KEY_WINDOW) {
        if (part->key_lo < 0 || part->key_hi <= part->key_lo || part->key_hi > L) return BDLM_ERR_INVALID_ARG;
        const bool all_rows = part->q_lo == 0 && part->q_hi == 0;
        if (!all_rows && (part->q_lo < 0 || part->q_hi <= part->q_lo || part->q_hi > L)) return BDLM_ERR_INVALID_ARG;
        lay->mode = MODE_WINDOW;
        lay->kw_lo = (int)part->key_lo;
        lay->kw_hi = (int)part->key_hi;
        lay->q_lo = all_rows ? 0 : (int)part->q_lo;
        lay->q_hi = all_rows ? (int)L : (int)part->q_hi;
        cm->mode = MODE_WINDOW;
        cm->Lq = lay->q_hi - lay->q_lo;
        cm->Lk = part->key_hi - part->key_lo;
    } else {
        if (part->q_lo != 0 || part->q_hi != 0) return BDLM_ERR_INVALID_ARG;  // row ranges are for windows
        // B rows per listed block (a short last block is padded to B)
        const long long nbk = (n + block - 1) / block;
        if (!part->q_blocks || part->n_q_blocks <= 0 || part->n_q_blocks > nbk) return BDLM_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(part->q_blocks) & 3u) return BDLM_ERR_INVALID_ARG;
        lay->mode = MODE_GROUP;
        lay->blocks = part->q_blocks;
        lay->n_blocks = part->n_q_blocks;
        cm->mode = MODE_GROUP;
        cm->Lq = (long long)part->n_q_blocks * block;
        cm->Lk = n + cm->Lq;
    }
    return BDLM_OK;
}

float pick_scale(float s, int d) { return s > 0.f ? s : 1.0f / std::sqrt((float)d); }

}  // namespace

extern "C" {

size_t bdlm_attn_fwd_workspace_bytes(int64_t L, int32_t heads, int32_t head_dim, int32_t n_docs) {
    if (L <= 0 || L > kMaxRows || heads <= 0 || (head_dim != 64 && head_dim != 128)) return 0;
    return sched_bytes(L, n_docs);
}

size_t bdlm_attn_bwd_workspace_bytes(int64_t L, int32_t heads, int32_t head_dim, int32_t n_docs) {
    if (L <= 0 || L > kMaxRows || heads <= 0 || (head_dim != 64 && head_dim != 128)) return 0;
    size_t b = sched_bytes(L, n_docs);
    b += round_up((size_t)L * heads * sizeof(float), 256);
    b += round_up((size_t)L * heads * head_dim * sizeof(float), 256);
    return b;
}

int bdlm_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t L, int32_t block,
                  int32_t heads, int32_t kv_heads, int32_t head_dim, const int32_t* cu_seqlens, int32_t n_docs,
                  float softmax_scale, const bdlm_partial* part, void* workspace, size_t workspace_bytes,
                  bdlm_stream_t stream) {
    g_launches = 0;
    Layout lay;
    Common cm{};
    int st = check_common(q, k, v, L, block, heads, kv_heads, head_dim, cu_seqlens, n_docs, part, &lay, &cm);
    if (st != BDLM_OK) return st;
    if (!o || !lse || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return BDLM_ERR_INVALID_ARG;
    const int kind = part ? part->kind : BDLM_PART_NONE;
    const int flags = part ? part->flags : 0;
    const int o_dtype = part ? part->o_dtype : BDLM_BF16;
    if (flags & ~BDLM_PART_ACCUMULATE) return BDLM_ERR_INVALID_ARG;
    if ((flags & BDLM_PART_ACCUMULATE) && kind != BDLM_PART_KEY_WINDOW) return BDLM_ERR_INVALID_ARG;
    if (o_dtype != BDLM_BF16 && o_dtype != BDLM_F32) return BDLM_ERR_INVALID_ARG;
    if (o_dtype == BDLM_F32 && kind == BDLM_PART_NONE) return BDLM_ERR_INVALID_ARG;
    const int docs = cu_seqlens ? n_docs : 1;
    if (!workspace || !aligned256(workspace)) return BDLM_ERR_WORKSPACE;
    if (workspace_bytes < bdlm_attn_fwd_workspace_bytes(L, heads, head_dim, docs)) return BDLM_ERR_WORKSPACE;
    const int sms = num_sms();
    if (sms <= 0) return BDLM_ERR_CUDA;

    WsCarve ws = carve(workspace, L, docs, heads, head_dim, false);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    launch_enumerate(lay, kFwdTileRows, kFwdKeyTile, 0, ws, s);
    if (cudaGetLastError() != cudaSuccess) return BDLM_ERR_CUDA;
    int launches = 1;

    FwdArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.v = static_cast<const __nv_bfloat16*>(v);
    a.o = o_dtype == BDLM_F32 ? nullptr : static_cast<__nv_bfloat16*>(o);
    a.o_f32 = o_dtype == BDLM_F32 ? static_cast<float*>(o) : nullptr;
    a.lse = lse;
    a.accumulate = (flags & BDLM_PART_ACCUMULATE) ? 1 : 0;
    a.lay = lay;
    a.H = heads;
    a.Hk = kv_heads;
    a.G = heads / kv_heads;
    a.D = head_dim;
    a.scale_log2 = pick_scale(softmax_scale, head_dim) * 1.4426950408889634f;
    a.Lq = cm.Lq;
    a.Lk = cm.Lk;
    a.table = ws.table;
    a.hdr = ws.hdr;
    if (launch_fwd_tc(a, ws.ranges, sms, s, &launches) != cudaSuccess) return BDLM_ERR_CUDA;
    g_launches = launches;
    return BDLM_OK;
}

size_t bdlm_attn_fwd_tasks_workspace_bytes(const bdlm_task* tasks, int32_t n_tasks) {
    const long long mt = tasks_max_tiles(tasks, n_tasks, false);
    if (mt < 0) return 0;
    return sched_bytes_mt(mt) + round_up((size_t)n_tasks * sizeof(TaskRec), 256);
}

size_t bdlm_attn_bwd_tasks_workspace_bytes(const bdlm_task* tasks, int32_t n_tasks, int64_t L, int32_t heads,
                                           int32_t head_dim) {
    const long long mt = tasks_max_tiles(tasks, n_tasks, true);
    if (mt < 0 || L <= 0 || L > kMaxRows || heads <= 0 || (head_dim != 64 && head_dim != 128)) return 0;
    size_t b = sched_bytes_mt(mt);
    b += round_up((size_t)L * heads * sizeof(float), 256);
    b += round_up((size_t)L * heads * head_dim * sizeof(float), 256);
    return b + round_up((size_t)n_tasks * sizeof(TaskRec), 256);
}

int bdlm_attn_fwd_tasks(const void* q, const void* k, const void* v, void* o, float* lse, int64_t L, int32_t block,
                        int32_t heads, int32_t kv_heads, int32_t head_dim, float softmax_scale,
                        const bdlm_task* tasks, int32_t n_tasks, int32_t n_slots, int32_t o_dtype, void* workspace,
                        size_t workspace_bytes, bdlm_stream_t stream) {
    g_launches = 0;
    if (!q || !k || !v || !o || !lse || !tasks) return BDLM_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return BDLM_ERR_INVALID_ARG;
    if (L <= 0 || L > kMaxRows || block <= 0 || heads <= 0 || kv_heads <= 0 || heads % kv_heads != 0)
        return BDLM_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return BDLM_ERR_UNSUPPORTED;
    if (o_dtype != BDLM_BF16 && o_dtype != BDLM_F32) return BDLM_ERR_INVALID_ARG;
    std::vector<TaskRec> rec;
    long long max_n = 1;
    const int st = check_tasks(tasks, n_tasks, L, n_slots, false, &rec, &max_n);
    if (st != BDLM_OK) return st;
    if (!workspace || !aligned256(workspace)) return BDLM_ERR_WORKSPACE;
    if (workspace_bytes < bdlm_attn_fwd_tasks_workspace_bytes(tasks, n_tasks)) return BDLM_ERR_WORKSPACE;
    const int sms = num_sms();
    if (sms <= 0) return BDLM_ERR_CUDA;

    WsCarve ws = carve_mt(workspace, tasks_max_tiles(tasks, n_tasks, false), L, heads, head_dim, false, n_tasks);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int launches = launch_task_upload(rec.data(), n_tasks, ws.tasks, s);
    Layout lay;
    std::memset(&lay, 0, sizeof(lay));
    lay.mode = MODE_TASKS;
    lay.B = block;
    lay.n = (int)max_n;  // the longest sequence bounds every tile's cost
    lay.n_docs = 1;
    lay.L = L;
    lay.tasks = ws.tasks;
    lay.n_tasks = n_tasks;
    launch_enumerate(lay, kFwdTileRows, kFwdKeyTile, 0, ws, s);
    if (cudaGetLastError() != cudaSuccess) return BDLM_ERR_CUDA;
    ++launches;

    FwdArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.v = static_cast<const __nv_bfloat16*>(v);
    a.o = o_dtype == BDLM_F32 ? nullptr : static_cast<__nv_bfloat16*>(o);
    a.o_f32 = o_dtype == BDLM_F32 ? static_cast<float*>(o) : nullptr;
    a.lse = lse;
    a.accumulate = 0;
    a.lay = lay;
    a.H = heads;
    a.Hk = kv_heads;
    a.G = heads / kv_heads;
    a.D = head_dim;
    a.scale_log2 = pick_scale(softmax_scale, head_dim) * 1.4426950408889634f;
    a.Lq = L;
    a.Lk = L;
    a.table = ws.table;
    a.hdr = ws.hdr;
    if (launch_fwd_tc(a, ws.ranges, sms, s, &launches) != cudaSuccess) return BDLM_ERR_CUDA;
    g_launches = launches;
    return BDLM_OK;
}

int bdlm_attn_bwd_tasks(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                        void* dq, void* dk, void* dv, int64_t L, int32_t block, int32_t heads, int32_t kv_heads,
                        int32_t head_dim, float softmax_scale, const bdlm_task* tasks, int32_t n_tasks,
                        int32_t n_slots, void* workspace, size_t workspace_bytes, bdlm_stream_t stream) {
    g_launches = 0;
    if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !tasks) return BDLM_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return BDLM_ERR_INVALID_ARG;
    if (L <= 0 || L > kMaxRows || block <= 0 || heads <= 0 || kv_heads <= 0 || heads % kv_heads != 0)
        return BDLM_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return BDLM_ERR_UNSUPPORTED;
    std::vector<TaskRec> rec;
    long long max_n = 1;
    const int st = check_tasks(tasks, n_tasks, L, n_slots, true, &rec, &max_n);
    if (st != BDLM_OK) return st;
    if (!workspace || !aligned256(workspace)) return BDLM_ERR_WORKSPACE;
    if (workspace_bytes < bdlm_attn_bwd_tasks_workspace_bytes(tasks, n_tasks, L, heads, head_dim))
        return BDLM_ERR_WORKSPACE;
    const int sms = num_sms();
    if (sms <= 0) return BDLM_ERR_CUDA;

    WsCarve ws = carve_mt(workspace, tasks_max_tiles(tasks, n_tasks, true), L, heads, head_dim, true, n_tasks);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int launches = launch_task_upload(rec.data(), n_tasks, ws.tasks, s);
    Layout lay;
    std::memset(&lay, 0, sizeof(lay));
    lay.mode = MODE_TASKS;
    lay.B = block;
    lay.n = (int)max_n;  // the longest sequence bounds every tile's cost
    lay.n_docs = 1;
    lay.L = L;
    lay.tasks = ws.tasks;
    lay.n_tasks = n_tasks;
    launch_enumerate(lay, kBwdKeyTile, kBwdQTile, 1, ws, s);
    if (cudaGetLastError() != cudaSuccess) return BDLM_ERR_CUDA;
    ++launches;

    BwdArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.v = static_cast<const __nv_bfloat16*>(v);
    a.o = static_cast<const __nv_bfloat16*>(o);
    a.lse = lse;
    a.dO = static_cast<const __nv_bfloat16*>(dO);
    a.dq = static_cast<__nv_bfloat16*>(dq);
    a.dk = static_cast<__nv_bfloat16*>(dk);
    a.dv = static_cast<__nv_bfloat16*>(dv);
    a.Dsum = ws.D;
    a.dqacc = ws.dqacc;
    a.lay = lay;
    a.H = heads;
    a.Hk = kv_heads;
    a.G = heads / kv_heads;
    a.D = head_dim;
    a.scale = pick_scale(softmax_scale, head_dim);
    a.scale_log2 = a.scale * 1.4426950408889634f;
    a.Lq = L;
    a.Lk = L;
    a.table = ws.table;
    a.hdr = ws.hdr;
    if (launch_bwd(a, sms, s, &launches) != cudaSuccess) return BDLM_ERR_CUDA;
    g_launches = launches;
    return BDLM_OK;
}

int bdlm_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, int64_t L, int32_t block, int32_t heads, int32_t kv_heads,
                  int32_t head_dim, const int32_t* cu_seqlens, int32_t n_docs, float softmax_scale,
                  const bdlm_partial* part, void* workspace, size_t workspace_bytes, bdlm_stream_t stream) {
    g_launches = 0;
    Layout lay;
    Common cm{};
    int st = check_common(q, k, v, L, block, heads, kv_heads, head_dim, cu_seqlens, n_docs, part, &lay, &cm);
    if (st != BDLM_OK) return st;
    if (part && (part->flags != 0 || part->o_dtype != BDLM_BF16)) return BDLM_ERR_INVALID_ARG;  // forward-only fields
    if (!o || !lse || !dO || !dq || !dk || !dv) return BDLM_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return BDLM_ERR_INVALID_ARG;
    const int docs = cu_seqlens ? n_docs : 1;
    if (!workspace || !aligned256(workspace)) return BDLM_ERR_WORKSPACE;
    if (workspace_bytes < bdlm_attn_bwd_workspace_bytes(L, heads, head_dim, docs)) return BDLM_ERR_WORKSPACE;
    const int sms = num_sms();
    if (sms <= 0) return BDLM_ERR_CUDA;

    WsCarve ws = carve(workspace, L, docs, heads, head_dim, true);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    launch_enumerate(lay, kBwdKeyTile, kBwdQTile, 1, ws, s);
    if (cudaGetLastError() != cudaSuccess) return BDLM_ERR_CUDA;
    int launches = 1;

    BwdArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.v = static_cast<const __nv_bfloat16*>(v);
    a.o = static_cast<const __nv_bfloat16*>(o);
    a.lse = lse;
    a.dO = static_cast<const __nv_bfloat16*>(dO);
    a.dq = static_cast<__nv_bfloat16*>(dq);
    a.dk = static_cast<__nv_bfloat16*>(dk);
    a.dv = static_cast<__nv_bfloat16*>(dv);
    a.Dsum = ws.D;
    a.dqacc = ws.dqacc;
    a.lay = lay;
    a.H = heads;
    a.Hk = kv_heads;
    a.G = heads / kv_heads;
    a.D = head_dim;
    a.scale = pick_scale(softmax_scale, head_dim);
    a.scale_log2 = a.scale * 1.4426950408889634f;
    a.Lq = cm.Lq;
    a.Lk = cm.Lk;
    a.table = ws.table;
    a.hdr = ws.hdr;
    if (launch_bwd(a, sms, s, &launches) != cudaSuccess) return BDLM_ERR_CUDA;
    g_launches = launches;
    return BDLM_OK;
}

int bdlm_lse_merge(const void* const* partials, const float* const* lses, int32_t n_partials,
                   int32_t partial_dtype, int64_t rows, int32_t heads, int32_t head_dim, void* o, float* lse,
                   bdlm_stream_t stream) {
    g_launches = 0;
    if (!partials || !lses || !o || !lse) return BDLM_ERR_INVALID_ARG;
    if (n_partials < 1 || n_partials > 64) return BDLM_ERR_INVALID_ARG;
    if (rows <= 0 || rows > kMaxRows || heads <= 0 || heads > 256) return BDLM_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return BDLM_ERR_UNSUPPORTED;
    if (partial_dtype != BDLM_BF16 && partial_dtype != BDLM_F32) return BDLM_ERR_INVALID_ARG;
    if (!aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return BDLM_ERR_INVALID_ARG;
    MergeArgs a{};
    for (int p = 0; p < n_partials; ++p) {
        if (!partials[p] || !lses[p] || !aligned16(partials[p]) || (reinterpret_cast<uintptr_t>(lses[p]) & 3u))
            return BDLM_ERR_INVALID_ARG;
        if (partials[p] == o) return BDLM_ERR_INVALID_ARG;
        a.part[p] = partials[p];
        a.lse_in[p] = lses[p];
    }
    a.P = n_partials;
    a.f32 = partial_dtype == BDLM_F32;
    a.rows = rows;
    a.H = heads;
    a.D = head_dim;
    a.o = static_cast<__nv_bfloat16*>(o);
    a.lse = lse;
    int launches = 0;
    if (launch_merge(a, num_sms(), reinterpret_cast<cudaStream_t>(stream), &launches) != cudaSuccess)
        return BDLM_ERR_CUDA;
    g_launches = launches;
    return BDLM_OK;
}

int bdlm_read_error(const void* workspace, bdlm_stream_t stream) {
    if (!workspace) {  // the no-allocation forward's scratch on the current device
        void* p = nullptr;
        const int st = noalloc_scratch(&p);
        if (st != BDLM_OK) return st;
        workspace = p;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int word[2] = {0, 0};
    if (cudaMemcpyAsync(word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return BDLM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return BDLM_ERR_CUDA;
    return word[0];
}

const char* bdlm_status_string(int status) {
    switch (status) {
        case BDLM_OK: return "BDLM_OK";
        case BDLM_ERR_INVALID_ARG: return "BDLM_ERR_INVALID_ARG";
        case BDLM_ERR_UNSUPPORTED: return "BDLM_ERR_UNSUPPORTED";
        case BDLM_ERR_WORKSPACE: return "BDLM_ERR_WORKSPACE";
        case BDLM_ERR_CUDA: return "BDLM_ERR_CUDA";
        case BDLM_ERR_TIMEOUT: return "BDLM_ERR_TIMEOUT";
        case BDLM_ERR_DEVICE_CHECK: return "BDLM_ERR_DEVICE_CHECK";
        default: return "BDLM_ERR_UNKNOWN";
    }
}

int bdlm_last_launch_count(void) { return g_launches; }

}  // extern "C"
