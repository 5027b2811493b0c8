// fwd_tc.cu - BDLM attention forward on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in TMEM, operands staged by TMA).
//
// One persistent CTA per SM takes work items (128-row query tile, pair of
// query heads that share one kv head) from the ordered tile list. Both heads
// of a pair see the same keys under the same mask, so one K/V stream in
// shared memory feeds two 128-row MMA tiles. In a task list every tile
// carries its task, which gives its key window (through the row spans) and
// the output slot its rows are written to.
//
// Warp roles (384 threads, launched at 168 registers each):
//   warps 0-3  softmax group 0 (head h0), one TMEM lane = one query row each
//   warps 4-7  softmax group 1 (head h0 + 1)
//   warp  8    TMA producer: Q tiles once per item, K/V tiles into a 2-stage ring
//   warp  9    TMEM owner and MMA issuer (one thread)
//   warps 10-11 spare (they only give their registers away)
// Register budget: warps 8-11 drop to 56 registers and the eight softmax warps
// rise to 224: 8 x 224 + 4 x 56 = 12 x 168, and per SM sub-partition
// (warps w, w+4, w+8) 224 + 224 + 56 = 504 <= 512.
// TMEM (512 columns): S0 | S1 | O0 | O1; P_i (bf16) overwrites the first 64
// columns of S_i after the softmax group has read S_i into registers.
// Per key tile j (128 keys):  S_i = Q_i K_j^T  ->  softmax_i  ->  O_i += P_i V_j.
// The next S_i is issued right behind O_i += P_i V_j: the tensor pipe runs a
// CTA's MMAs in issue order, so the PV MMA reads P_i before S_i overwrites
// it, and the softmax, which waits for S_i's commit, sees O_i complete (an
// MMA's commit covers every MMA issued before it) before it rescales O_i.
// The tensor pipe holds little more than the MMA it is running, so each wait,
// fence or commit of the issuing thread leaves it idle for about as long as
// that step takes. The issuer therefore waits once per key tile for K_j and
// V_j together (one barrier), once per head for the whole of P_i, and
// commits O_i only after the item's last key tile.
// A key tile with masked entries is masked in TMEM (-inf written over the
// entries) before the softmax reads it, so unmasked tiles run no mask code.
// Online softmax in fp32 registers, base 2, with a lazily moved offset: the
// running row offset changes only when the row max exceeds it by more than
// 2^8, and only then is the O row in TMEM rescaled.
// Every mbarrier wait is bounded (2 s); a timeout sets the workspace error
// word to BDLM_ERR_TIMEOUT and all roles drain out.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace bdlm {
namespace {

constexpr int BM = 128;  // query rows per tile (MMA M)
constexpr int BN = 128;  // keys per step (MMA N of S = Q K^T)
constexpr int kThreads = 384;
constexpr int kRegsSoftmax = 224;
constexpr int kRegsOther = 56;
constexpr int kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 2000000000ull;

template <int D>
struct Lay {
    static constexpr int kTile = BM * D * 2;       // bytes of a 128-row tile
    static constexpr int kChunk = BM * 128;        // bytes of a 64-column, 128-row swizzled chunk
    static constexpr int kQ0 = 0;
    static constexpr int kQ1 = kTile;
    static constexpr int kK = 2 * kTile;           // + stage * kTile
    static constexpr int kV = 4 * kTile;           // + stage * kTile
    static constexpr int kBytes = 6 * kTile + 1024;  // + alignment slack
};

// barrier slots
enum : int { B_Q = 0, B_KVFULL = 1, B_KVEMPTY = 3, B_S = 5, B_P = 7, B_O = 9, B_COUNT = 11 };

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ int key_start(const TileRange& R, int n1, int j) {
    return j < n1 ? R.r1_lo + j * BN : R.r2_lo + (j - n1) * BN;
}

struct ItemCtx {
    Tile T;
    TileRange R;
    int n1, nk;
    int kvh, h0;
    bool two;
    int q_row0;
};

// ---------------------------------------------------------------- producer
template <int D>
__device__ __forceinline__ void produce(const ItemCtx& c, uint32_t sbase, const uint64_t* bar,
                                        const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                                        uint32_t t_base, volatile int* abort) {
    using S = Lay<D>;
    constexpr int NC = D / 64;
    const uint32_t bq = tc::smem_addr(&bar[B_Q]);
    tc::mbar_arrive_expect_tx(bq, (c.two ? 2 : 1) * S::kTile);
    for (int ch = 0; ch < NC; ++ch) {
        tc::tma_load_3d(sbase + S::kQ0 + ch * S::kChunk, tq, bq, 64 * ch, c.h0, c.q_row0);
        if (c.two) tc::tma_load_3d(sbase + S::kQ1 + ch * S::kChunk, tq, bq, 64 * ch, c.h0 + 1, c.q_row0);
    }
    for (int j = 0; j < c.nk; ++j) {
        const uint32_t t = t_base + j, s = t & 1, ph = (t >> 1) & 1;
        if (!tc::mbar_wait(tc::smem_addr(&bar[B_KVEMPTY + s]), ph ^ 1, abort, kTimeoutNs)) return;
        const int k0 = key_start(c.R, c.n1, j);
        // K_j and V_j complete one barrier: the MMA issuer waits once per key tile
        const uint32_t bkv = tc::smem_addr(&bar[B_KVFULL + s]);
        tc::mbar_arrive_expect_tx(bkv, 2 * S::kTile);
        for (int ch = 0; ch < NC; ++ch)
            tc::tma_load_3d(sbase + S::kK + s * S::kTile + ch * S::kChunk, tk, bkv, 64 * ch, c.kvh, k0);
        for (int ch = 0; ch < NC; ++ch)
            tc::tma_load_3d(sbase + S::kV + s * S::kTile + ch * S::kChunk, tv, bkv, 64 * ch, c.kvh, k0);
    }
}

// --------------------------------------------------------------------- MMA
template <int D>
__device__ __forceinline__ void issue_mma(const ItemCtx& c, uint32_t sbase, const uint64_t* bar, uint32_t tmem,
                                          uint32_t t_base, uint32_t t_base1, uint32_t q_count,
                                          volatile int* abort) {
    using S = Lay<D>;
    constexpr uint32_t idesc_s = tc::idesc_bf16(BM, BN, 0);
    constexpr uint32_t idesc_o = tc::idesc_bf16(BM, D, 1);
    if (!tc::mbar_wait(tc::smem_addr(&bar[B_Q]), q_count & 1, abort, kTimeoutNs)) return;
    tc::tc_fence_after();
    const int nh = c.two ? 2 : 1;
    // operand descriptors of the shared-memory base, K-major (Q, K) and
    // MN-major (V); tiles, K slices and stages are constant offsets
    const uint64_t km = tc::sdesc_sw128(sbase, 16, 1024);
    const uint64_t mn = tc::sdesc_sw128(sbase, S::kChunk, 1024);
    // S_i = Q_i K_j^T into head i's S columns
    auto issue_s = [&](int i, uint32_t stage) {
        const uint64_t dK = tc::sdesc_add(km, S::kK + stage * S::kTile);
        const uint64_t dQ = tc::sdesc_add(km, i == 0 ? S::kQ0 : S::kQ1);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * S::kChunk + (k & 3) * 32;
            tc::mma_ss(tmem + 128 * i, tc::sdesc_add(dQ, off), tc::sdesc_add(dK, off), idesc_s, k > 0);
        }
        tc::mma_commit(tc::smem_addr(&bar[B_S + i]));
    };
    if (c.nk == 0) return;
    {
        const uint32_t t = t_base, s = t & 1, ph = (t >> 1) & 1;
        if (!tc::mbar_wait(tc::smem_addr(&bar[B_KVFULL + s]), ph, abort, kTimeoutNs)) return;
        tc::tc_fence_after();
        for (int i = 0; i < nh; ++i) issue_s(i, s);
    }
    for (int j = 0; j < c.nk; ++j) {
        const uint32_t t = t_base + j, s = t & 1, ph = (t >> 1) & 1;
        const uint32_t tn = t + 1, sn = tn & 1, phn = (tn >> 1) & 1;
        const uint64_t dV = tc::sdesc_add(mn, S::kV + s * S::kTile);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (i >= nh) break;
            const uint32_t ti = i == 0 ? t : t_base1 + j;
            const uint32_t tS = tmem + 128 * i, tO = tmem + 256 + D * i;
            // one wait for the whole of P_i: every wait of this thread leaves
            // the tensor pipe idle for as long as it takes
            if (!tc::mbar_wait(tc::smem_addr(&bar[B_P + i]), ti & 1, abort, kTimeoutNs)) return;
            tc::tc_fence_after();
#pragma unroll
            for (int k = 0; k < BN / 16; ++k)
                tc::mma_ts(tO, tS + 8 * k, tc::sdesc_add(dV, 2048 * k), idesc_o, (j > 0 || k > 0) ? 1u : 0u);
            if (j + 1 == c.nk) tc::mma_commit(tc::smem_addr(&bar[B_O + i]));  // O_i complete
            if (i == nh - 1) tc::mma_commit(tc::smem_addr(&bar[B_KVEMPTY + s]));  // K_j, V_j read
            // S_i of the next key tile right behind PV_i: the tensor pipe runs
            // this CTA's MMAs in issue order, so it reads P_i before S_i
            // overwrites it, and its commit covers PV_i
            if (j + 1 < c.nk) {
                if (i == 0) {
                    if (!tc::mbar_wait(tc::smem_addr(&bar[B_KVFULL + sn]), phn, abort, kTimeoutNs)) return;
                    tc::tc_fence_after();
                }
                issue_s(i, sn);
            }
        }
    }
}

// ----------------------------------------------------------------- softmax
// One thread per query row of head h0 + i. Reads S_i, writes P_i (bf16) back
// into TMEM, keeps the row offset and sum, rescales O_i when the offset moves,
// and finally normalises O_i and stores o and lse. TMEM loads and stores are
// warp-collective, so every branch around them is warp-uniform.
template <int D>
__device__ __forceinline__ void softmax_rows(const ItemCtx& c, const FwdArgs& a, const uint64_t* bar, uint32_t tmem,
                                             int i, uint32_t tb, uint32_t o_count, volatile int* abort,
                                             const int* item_p) {
    const int row = threadIdx.x & 127;
    const uint32_t lane_base = (uint32_t)(32 * ((threadIdx.x >> 5) & 3)) << 16;
    const uint32_t tS = tmem + i * 128 + lane_base;
    const uint32_t tO = tmem + 256 + i * D + lane_base;
    const int h = c.h0 + i;
    const Span sp = row_span(a.lay, c.T, row);
    const float sl2 = a.scale_log2;
    float m_use = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < c.nk; ++j) {
        const uint32_t t = tb + j;
        const bool got = tc::mbar_wait(tc::smem_addr(&bar[B_S + i]), t & 1, abort, kTimeoutNs);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc::tc_fence_after();
        const int k0 = key_start(c.R, c.n1, j);
        const bool full = j < c.n1 && k0 >= c.R.full_lo && k0 + BN <= c.R.full_hi;  // warp-uniform
        if (!full) {
            // a tile with masked entries: write -inf over them in TMEM first,
            // so that the path of unmasked tiles carries no mask code
            const RelInterval ri = range_interval(sp, j < c.n1, k0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t m[32];
                tc::tmem_ld32(tS + 32 * q, m);
                tc::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (!rel_sees(ri, 32 * q + e)) m[e] = 0xff800000u;  // -inf
                tc::tmem_st32(tS + 32 * q, m);
            }
            tc::tmem_st_wait();
        }
        uint32_t r[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tc::tmem_ld32(tS + 32 * q, r[q]);
        tc::tmem_ld_wait();
        float x[128];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int e = 0; e < 32; ++e) x[32 * q + e] = __uint_as_float(r[q][e]);
        // row max, four independent chains of three-input max
        float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
        for (int e = 4; e < 128; e += 8) {
            mx0 = tc::fmax3(mx0, x[e], x[e + 1]);
            mx1 = tc::fmax3(mx1, x[e + 2], x[e + 3]);
            mx2 = tc::fmax3(mx2, x[e + 4], x[e + 5]);
            mx3 = tc::fmax3(mx3, x[e + 6], x[e + 7]);
        }
        const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
        const bool move = mx > m_use + 8.0f;
        float alpha = 1.f;
        if (move) {
            alpha = ex2f(m_use - mx);
            l *= alpha;
            m_use = mx;
        }
        if (j > 0 && __any_sync(0xffffffffu, move)) {
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tc::tmem_ld32(tO + 32 * q, o);
                tc::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tc::tmem_st32(tO + 32 * q, o);
            }
        }
        const float m_eff = m_use == -INFINITY ? 0.f : m_use;
        // p = exp2(x * scale * log2 e - m) on packed pairs; row sum in two lanes
        const float2 sl2x2 = make_float2(sl2, sl2), nm2 = make_float2(-m_eff, -m_eff);
        float2 sum2 = make_float2(0.f, 0.f);
        uint32_t pa[32], pb[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float2 y = tc::fma2(make_float2(x[2 * e], x[2 * e + 1]), sl2x2, nm2);
            const float2 p = make_float2(ex2f(y.x), ex2f(y.y));
            sum2 = tc::add2(sum2, p);
            pa[e] = pack2(p.x, p.y);
        }
        tc::tmem_st32(tS, pa);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float2 y = tc::fma2(make_float2(x[64 + 2 * e], x[64 + 2 * e + 1]), sl2x2, nm2);
            const float2 p = make_float2(ex2f(y.x), ex2f(y.y));
            sum2 = tc::add2(sum2, p);
            pb[e] = pack2(p.x, p.y);
        }
        tc::tmem_st32(tS + 32, pb);
        l += sum2.x + sum2.y;
        tc::tmem_st_wait();
        tc::tc_fence_before();
        __syncwarp();  // the warp's P columns are all in TMEM; one arrival per warp
        if ((threadIdx.x & 31) == 0) tc::mbar_arrive(tc::smem_addr(&bar[B_P + i]));
    }
    if (ok && c.nk > 0) {
        const bool got = tc::mbar_wait(tc::smem_addr(&bar[B_O + i]), o_count & 1, abort, kTimeoutNs);
        ok = __all_sync(0xffffffffu, got);
        tc::tc_fence_after();
    }
    const bool have_o = ok && c.nk > 0;  // warp-uniform
    const bool store = row < c.T.nrows;
    // o [slots, Lq, H, D], lse [slots, H, Lq]; a task list's tile takes the
    // slot of its task (looked up again from the item number, which stays in
    // shared memory until every role has finished the item)
    int slot = 0;
    if (a.lay.mode == MODE_TASKS) {
        const int n_pairs = a.Hk * ((a.G + 1) / 2);
        slot = ld_ro(&a.lay.tasks[ld_ro(&a.table[*item_p / n_pairs].task)].slot);
    }
    const long long ooff = ((long long)slot * a.Lq + c.q_row0 + row) * ((long long)a.H * D) + (long long)h * D;
    const long long lidx = ((long long)slot * a.H + h) * a.Lq + c.q_row0 + row;
    // this call's row: lse in base 2, o = (unnormalised O) * cw
    const float l2w = l > 0.f ? m_use + __log2f(l) : -INFINITY;
    float cw = l > 0.f ? 1.f / l : 0.f, ca = 0.f, l2out = l2w;
    bool write = store;
    if (a.accumulate && store) {
        // running merge with the stored result of earlier windows (log-sum-exp
        // weights in fp32); a window the row cannot see leaves it unchanged
        const float l2a = a.lse[lidx] * 1.4426950408889634f;
        if (l2w == -INFINITY) {
            write = false;
        } else if (l2a != -INFINITY) {
            const float mx = fmaxf(l2a, l2w);
            const float wa = ex2f(l2a - mx), ww = ex2f(l2w - mx);
            const float rz = 1.f / (wa + ww);
            ca = wa * rz;
            cw *= ww * rz;
            l2out = mx + __log2f(wa + ww);
        }
    }
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
        uint32_t o[32];
        if (have_o) {
            tc::tmem_ld32(tO + 32 * q, o);
            tc::tmem_ld_wait();
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (!write) continue;
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(o[e]) * cw;
        if (a.o_f32) {
            float4* dst = reinterpret_cast<float4*>(a.o_f32 + ooff + 32 * q);
            if (ca != 0.f) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 t = dst[e];
                    v[4 * e] = fmaf(ca, t.x, v[4 * e]);
                    v[4 * e + 1] = fmaf(ca, t.y, v[4 * e + 1]);
                    v[4 * e + 2] = fmaf(ca, t.z, v[4 * e + 2]);
                    v[4 * e + 3] = fmaf(ca, t.w, v[4 * e + 3]);
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        } else {
            uint4* dst = reinterpret_cast<uint4*>(a.o + ooff + 32 * q);
            if (ca != 0.f) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint4 t = dst[e];
                    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        v[8 * e + 2 * u] = fmaf(ca, __uint_as_float(w[u] << 16), v[8 * e + 2 * u]);
                        v[8 * e + 2 * u + 1] = fmaf(ca, __uint_as_float(w[u] & 0xffff0000u), v[8 * e + 2 * u + 1]);
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e)
                dst[e] = make_uint4(pack2(v[8 * e], v[8 * e + 1]), pack2(v[8 * e + 2], v[8 * e + 3]),
                                    pack2(v[8 * e + 4], v[8 * e + 5]), pack2(v[8 * e + 6], v[8 * e + 7]));
        }
    }
    if (write) a.lse[lidx] = l2out == -INFINITY ? -INFINITY : l2out * 0.69314718055994531f;
}

// ------------------------------------------------------------------ kernel
__device__ __forceinline__ void named_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

__device__ __forceinline__ ItemCtx decode(const FwdArgs& a, const TileRange* ranges, int item, int n_pairs,
                                          int per_kv) {
    ItemCtx c;
    const int ti = item / n_pairs, pr = item % n_pairs;
    c.T = a.table[ti];
    c.R = ranges[ti];
    c.kvh = pr / per_kv;
    const int hp = pr % per_kv;
    c.h0 = c.kvh * a.G + 2 * hp;
    c.two = 2 * hp + 1 < a.G;
    c.n1 = (c.R.r1_hi - c.R.r1_lo + BN - 1) / BN;
    c.nk = c.n1 + (c.R.r2_hi - c.R.r2_lo + BN - 1) / BN;
    c.q_row0 = q_row_of(a.lay, c.T, c.T.pos0);
    return c;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdArgs a, const TileRange* __restrict__ ranges) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = tc::smem_addr(smem);
    __shared__ __align__(8) uint64_t bar[B_COUNT];
    __shared__ uint32_t s_tmem;
    __shared__ int s_item;
    __shared__ int s_abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        s_abort = 0;
        tc::mbar_init(tc::smem_addr(&bar[B_Q]), 1);
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(tc::smem_addr(&bar[B_KVFULL + s]), 1);
            tc::mbar_init(tc::smem_addr(&bar[B_KVEMPTY + s]), 1);
            tc::mbar_init(tc::smem_addr(&bar[B_S + s]), 1);
            tc::mbar_init(tc::smem_addr(&bar[B_P + s]), 4);  // lane 0 of each softmax warp
            tc::mbar_init(tc::smem_addr(&bar[B_O + s]), 1);
        }
        tc::fence_barrier_init();
    }
    if (warp == 9) {
        tc::tmem_alloc(tc::smem_addr(&s_tmem), kTmemCols);
        tc::tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* abort = &s_abort;

    const int per_kv = (a.G + 1) / 2;
    const int n_pairs = a.Hk * per_kv;
    const int n_items = a.hdr->n_tiles * n_pairs;
    uint32_t t_base = 0, t_base1 = 0, q_count = 0;
    // Two register regions: each role branch runs its own copy of the item
    // loop; the branches meet at named barrier 1 (all 384 threads) twice per item.
    if (warp >= 8) {
        tc::regs_dec<kRegsOther>();
        for (;;) {
            named_sync();
            if (tid == 256) s_item = *abort ? n_items : atomicAdd(&a.hdr->counter, 1);
            named_sync();
            const int item = s_item;
            if (item >= n_items) break;
            const ItemCtx c = decode(a, ranges, item, n_pairs, per_kv);
            if (warp == 8 && lane == 0 && c.nk > 0) produce<D>(c, sbase, bar, &tm_q, &tm_k, &tm_v, t_base, abort);
            if (warp == 9 && lane == 0 && c.nk > 0)
                issue_mma<D>(c, sbase, bar, tmem, t_base, t_base1, q_count, abort);
            t_base += c.nk;
            if (c.two) t_base1 += c.nk;
            if (c.nk > 0) ++q_count;
        }
    } else {
        tc::regs_inc<kRegsSoftmax>();
        const int wg = warp >> 2;
        uint32_t o_count = 0;  // items with key tiles that this head slot has finished
        for (;;) {
            named_sync();
            named_sync();
            const int item = s_item;
            if (item >= n_items) break;
            const ItemCtx c = decode(a, ranges, item, n_pairs, per_kv);
            if (wg == 0 || c.two) {
                softmax_rows<D>(c, a, bar, tmem, wg, wg == 0 ? t_base : t_base1, o_count, abort, &s_item);
                if (c.nk > 0) ++o_count;
            }
            t_base += c.nk;
            if (c.two) t_base1 += c.nk;
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && s_abort) set_error(a.hdr, DEV_TIMEOUT, blockIdx.x);
}

// ------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// [rows, heads, D] bf16 tensor as a 3-D map (D, heads, rows) with 64 x 1 x 128 boxes, 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, int D, int heads, long long rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)BM};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_tc(const FwdArgs& a, const TileRange* ranges, int num_sms, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, D, a.H, a.Lq) || !make_map(&mk, a.k, D, a.Hk, a.Lk) || !make_map(&mv, a.v, D, a.Hk, a.Lk))
        return cudaErrorInvalidValue;
    constexpr int smem = Lay<D>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    fwd_tc_kernel<D><<<num_sms, kThreads, smem, st>>>(mq, mk, mv, a, ranges);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdArgs& a, const TileRange* ranges, int num_sms, cudaStream_t st, int* launches) {
    cudaError_t e = a.D == 128 ? launch_tc<128>(a, ranges, num_sms, st) : launch_tc<64>(a, ranges, num_sms, st);
    if (e == cudaSuccess) ++*launches;
    return e;
}

}  // namespace bdlm
