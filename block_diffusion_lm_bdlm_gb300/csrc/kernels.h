// kernels.h - internal launch interface between the C ABI and the kernels.
#pragma once

#include "common.cuh"

namespace bdlm {

// Workspace carve-up (all pointers inside the caller's workspace).
struct WsCarve {
    WsHeader* hdr;
    Tile* table;    // ordered tiles
    Tile* tmp;      // unordered tiles (prologue scratch)
    int* cost;      // per-tile cost (prologue scratch)
    TileRange* ranges;   // key ranges of the ordered tiles (forward)
    TileRange* rng_tmp;  // key ranges of the unordered tiles (prologue scratch)
    TaskRec* tasks;      // task list (task-list forward)
    int max_tiles;
    float* D;       // backward: rowsum(dO * o), [H, L]
    float* dqacc;   // backward: fp32 dq accumulator, [L, H, d]
};

struct FwdArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    __nv_bfloat16* o;   // bf16 output (o_f32 == nullptr)
    float* o_f32;       // fp32 output of a partial (o == nullptr)
    float* lse;
    int accumulate;     // merge into the running (o, lse) instead of overwriting
    Layout lay;
    int H, Hk, G, D;
    float scale_log2;  // softmax scale * log2(e)
    long long Lq, Lk;  // rows of q and of k
    const Tile* table;
    WsHeader* hdr;
};

struct BwdArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const __nv_bfloat16* o;
    const float* lse;
    const __nv_bfloat16* dO;
    __nv_bfloat16* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    float* Dsum;
    float* dqacc;
    Layout lay;
    int H, Hk, G, D;
    float scale, scale_log2;
    long long Lq, Lk;  // rows of q (o, dO, dq, lse, D) and of k (v, dk, dv)
    const Tile* table;
    WsHeader* hdr;
};

struct MergeArgs {
    const void* part[64];
    const float* lse_in[64];
    int P;
    int f32;  // partials are fp32
    long long rows;
    int H, D;
    __nv_bfloat16* o;
    float* lse;
};

// Tile heights used by the kernels (the prologue enumerates in these units).
constexpr int kFwdTileRows = 128;  // tensor-core forward: 128-row query tiles
constexpr int kFwdKeyTile = 128;   // and 128-key steps
constexpr int kBwdKeyTile = 128;  // backward: 128-key items
constexpr int kBwdQTile = 128;    // and 128-row query steps

// Task records per upload launch (kernel parameters stay under 32 KB).
constexpr int kTaskUploadChunk = 960;
int launch_task_upload(const TaskRec* host, int n, TaskRec* dst, cudaStream_t st);  // returns launches
void launch_enumerate(const Layout& lay, int tile_rows, int key_tile, int kind, const WsCarve& ws,
                      cudaStream_t st);
cudaError_t launch_fwd_tc(const FwdArgs& a, const TileRange* ranges, int num_sms, cudaStream_t st, int* launches);
cudaError_t launch_bwd(const BwdArgs& a, int num_sms, cudaStream_t st, int* launches);
cudaError_t launch_bwd_tc_main(const BwdArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_merge(const MergeArgs& a, int num_sms, cudaStream_t st, int* launches);

// Device address of the no-allocation forward's fixed scratch on the current
// device (a bdlm_status; looked up again after the context changes).
int noalloc_scratch(void** out);

}  // namespace bdlm
