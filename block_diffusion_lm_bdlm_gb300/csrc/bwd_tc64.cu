// bwd_tc64.cu - (64-row steps) BDLM attention backward main kernel on the 5th-generation
// tensor cores (head_dim 128).
//
// Key-major: one work item = (128-key tile, kv head). The item loops over the
// G query heads of the kv head and, for each, over the 64-row query steps
// that see the key tile (a clean key tile is seen by the clean rows from its
// block on and by the corrupted rows of later blocks; a corrupted key tile
// only by its own blocks' corrupted rows). Per step:
//   S^T  = K Q^T          (M 128 keys, N 64 rows, K = d)      -> TMEM
//   dP^T = V dO^T                                              -> TMEM
//   P^T  = exp2(S^T*scale*log2e - lse*log2e), dS^T = P^T (dP^T - D)
//          (compute warps; P^T and dS^T go to their own TMEM columns as bf16
//          for dV and dK, and dS^T also to shared memory for dQ^T)
//   dV  += P^T dO         (A from TMEM)                        -> TMEM
//   dK  += dS^T Q         (A from TMEM)                        -> TMEM
//   dQ^T = K^T dS^T       (M = d, N 64 rows, K 128 keys)       -> TMEM
//          read out, scaled, staged in shared memory and added into the fp32
//          dq accumulator with one TMA reduce-add per step.
// dK and dV stay in TMEM for the whole item (no atomics: the item owns its
// keys for all G heads) and are written once, as bf16, at the end.
//
// Warp roles (448 threads):
//   warps 0-7   P/dS groups: one TMEM lane = one key row; group g (warps
//               4g..4g+3) takes query columns 32g..32g+31 of a step. The mask
//               is analytic: for one key, the rows of a step that see it form
//               one interval (later clean blocks / later corrupted blocks for a
//               clean key, its own corrupted block for a corrupted key).
//   warps 8-11  dq group: reads dQ^T (lane = d) out to the TMA reduce-add
//               through a double-buffered staging tile, and writes dK and dV
//               at the end of an item
//   warp  12    loader: TMA for K, V, Q, dO; plain loads for lse and D; 3-stage
//               ring for the per-step inputs
//   warp  13    TMEM owner and MMA issuer (one thread). Per step s it issues
//              S^T(s+1) and dP^T(s+1) as soon as the P/dS warps have read
//              S^T(s) and dP^T(s) out of TMEM, then dV(s) and dK(s) once
//              P/dS(s) is done, then dQ^T(s): the next step's S^T and dP^T run
//              on the tensor pipe while P/dS(s) computes.
// TMEM columns: dK [0,128) | dV [128,256) | S^T [256,320) | dP^T [320,384) |
// P^T [384,416) | dQ^T [416,480) | dS^T [480,512). dS^T in shared memory is
// double buffered. Because P^T and dS^T do not alias S^T and dP^T, S^T and
// dP^T are free once loaded (barrier B_LD); P^T and dS^T of step s+1 are
// written only after dV(s) and dK(s) completed (the stage's B_QDE commit).
// The shared-memory copy of dS^T has its own barrier, needed only by dQ^T;
// tcgen05 commit order covers the rest (an MMA's commit also covers every MMA
// issued before it).
// Every mbarrier wait is bounded (2 s).
#include <cuda.h>

#include <cstdlib>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace bdlm {
namespace {

constexpr int D = 128;
constexpr int BN = 128;  // keys per item
constexpr int BQ = 64;   // query rows per step
constexpr int kThreads = 448;
constexpr int kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 2000000000ull;

constexpr uint32_t TDK = 0, TDV = 128, TS = 256, TDP = 320, TP = 384, TDQ = 416, TDS = 480;
constexpr int kStages = 3;

// dynamic shared memory (1024-aligned offsets)
constexpr int kKV = BN * D * 2;     // 32 KB: K or V tile, two 64-column chunks of 16 KB
constexpr int kQT = BQ * D * 2;     // 16 KB: Q or dO tile, two chunks of 8 KB
constexpr int kST = BN * BQ * 2;    // 16 KB: dS^T [128 keys][64 rows] bf16, 128-byte swizzled rows
constexpr int kHalfRows = BQ / 2;   // dq staging holds half a step: [32 rows][128] fp32
constexpr int SM_K = 0;
constexpr int SM_V = SM_K + kKV;
constexpr int SM_Q = SM_V + kKV;                // + stage * kQT
constexpr int SM_O = SM_Q + kStages * kQT;      // + stage * kQT
constexpr int SM_S = SM_O + kStages * kQT;      // + buffer * kST
constexpr int kStg = kHalfRows * D * 4;  // 16 KB per staging buffer
constexpr int SM_STG = SM_S + 2 * kST;     // + buffer * kStg
constexpr int kSmemBytes = SM_STG + 2 * kStg + 1024;

enum : int {
    B_KV = 0, B_QDF = 1, B_QDE = 4, B_S = 7, B_DP = 8, B_SM = 9, B_SS = 10 /* x2, by step parity */, B_DQ = 12, B_DQF = 13,
    B_LD = 14, B_COUNT = 15
};

struct StepInfo {
    float nl2[BQ];   // -lse * log2(e) of the step's rows (0 beyond the step; those rows are masked)
    float dsum[BQ];  // D = rowsum(dO * o)
};

struct ItemCtx {
    Tile kt;
    int kvh, k0, kv_rows;
    int ra_lo, ra_hi, rb_lo, rb_hi, na, per_head, n_steps;
};

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
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_reduce_add_3d(const void* tmap, uint32_t src, int c0, int c1, int c2) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(tmap),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
// Barrier over the n threads of named barrier `id` that also ANDs a predicate,
// so that a decision to stop is taken by all of them together.
__device__ __forceinline__ bool named_and(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Item -> (key tile, kv head). Tiles are ordered heaviest first. By default
// (K = 1) the items of one tile (its kv heads) are consecutive, so the order
// is strictly heaviest first. For packed documents with many tiles the items
// go in blocks of K = gridDim.x / 2 tiles, kv head by kv head within a block
// (one wave of gridDim.x items spans two kv heads): measured on a GB300, this
// takes the 64-document packed backward from 93.3 to 85.1 ms, while single
// long sequences ran about 1 % faster with K = 1 (their DRAM traffic drops
// about 4x with the blocks, but they are not bound by it).
__device__ __forceinline__ ItemCtx decode(const BwdArgs& a, int item) {
    ItemCtx c;
    const int nt = a.hdr->n_tiles;
    const bool packed = a.lay.mode == MODE_FULL && a.lay.cu != nullptr;
    const int K = packed && nt >= 8 * (int)gridDim.x ? (int)gridDim.x / 2 : 1;
    const int per = K * a.Hk;
    const int ib = item / per, ir = item % per, kb = imin(K, nt - ib * K);
    c.kt = a.table[ib * K + ir % kb];
    c.kvh = ir / kb;
    c.k0 = key_row0(a.lay, c.kt);
    c.kv_rows = c.kt.nrows;
    const KeyRows r = key_tile_rows(a.lay, c.kt);
    c.ra_lo = r.a_lo;
    c.ra_hi = r.a_hi;
    c.rb_lo = r.b_lo;
    c.rb_hi = r.b_hi;
    c.na = (c.ra_hi - c.ra_lo + BQ - 1) / BQ;
    const int nb = (c.rb_hi - c.rb_lo + BQ - 1) / BQ;
    c.per_head = c.na + nb;
    c.n_steps = c.per_head * a.G;
    return c;
}

// query rows of step s: head, first document position, valid rows
__device__ __forceinline__ void step_rows(const ItemCtx& c, const BwdArgs& a, int s, int* h, int* p0, int* nrows) {
    const int hh = s / c.per_head, rem = s % c.per_head;
    *h = c.kvh * a.G + hh;
    *p0 = rem < c.na ? c.ra_lo + rem * BQ : c.rb_lo + (rem - c.na) * BQ;
    const int hi = rem < c.na ? c.ra_hi : c.rb_hi;
    *nrows = imin(BQ, hi - *p0);
}

// ---------------------------------------------------------------- loader
__device__ __forceinline__ void load_item(const ItemCtx& c, const BwdArgs& a, uint32_t sbase, const uint64_t* bar,
                                          StepInfo* info, const CUtensorMap* tk, const CUtensorMap* tv,
                                          const CUtensorMap* tq, const CUtensorMap* tdo, uint32_t ts_base,
                                          volatile int* abort) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        const uint32_t bkv = tc::smem_addr(&bar[B_KV]);
        tc::mbar_arrive_expect_tx(bkv, 2 * kKV);
        for (int ch = 0; ch < 2; ++ch) {
            tc::tma_load_3d(sbase + SM_K + ch * (kKV / 2), tk, bkv, 64 * ch, c.kvh, c.k0);
            tc::tma_load_3d(sbase + SM_V + ch * (kKV / 2), tv, bkv, 64 * ch, c.kvh, c.k0);
        }
    }
    for (int s = 0; s < c.n_steps; ++s) {
        const uint32_t ts = ts_base + s, st = ts % kStages, ph = (ts / kStages) & 1;
        const bool got = tc::mbar_wait(tc::smem_addr(&bar[B_QDE + st]), ph ^ 1, abort, kTimeoutNs);
        if (!__all_sync(0xffffffffu, got)) return;
        int h, p0, nrows;
        step_rows(c, a, s, &h, &p0, &nrows);
        const int qr0 = q_row_of(a.lay, c.kt, p0);
        const uint32_t bf = tc::smem_addr(&bar[B_QDF + st]);
        if (lane == 0) {
            mbar_expect_tx(bf, 2 * kQT);
            for (int ch = 0; ch < 2; ++ch) {
                tc::tma_load_3d(sbase + SM_Q + st * kQT + ch * (kQT / 2), tq, bf, 64 * ch, h, qr0);
                tc::tma_load_3d(sbase + SM_O + st * kQT + ch * (kQT / 2), tdo, bf, 64 * ch, h, qr0);
            }
        }
        // lse and D: plain loads (the loader runs steps ahead of the MMAs),
        // stored pre-scaled so that P/dS spends one FFMA per element before exp2
        StepInfo& inf = info[st];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int r = 2 * lane + u;
            float nl2 = 0.f, dd = 0.f;
            if (r < nrows) {
                const long long gi = (long long)h * a.Lq + qr0 + r;
                nl2 = -__ldg(a.lse + gi) * 1.4426950408889634f;
                dd = __ldg(a.Dsum + gi);
            }
            inf.nl2[r] = nl2;
            inf.dsum[r] = dd;
        }
        tc::mbar_arrive(bf);
    }
}

// ------------------------------------------------------------------- MMA
__device__ __forceinline__ bool mma_wait(const uint64_t* bar, int i, uint32_t parity, volatile int* abort) {
    if (!tc::mbar_wait(tc::smem_addr(&bar[i]), parity, abort, kTimeoutNs)) return false;
    tc::tc_fence_after();
    return true;
}

// Shared-memory descriptors of the operand tiles at stage / buffer 0; the MMA
// thread steps to K slices, stages and buffers with tc::sdesc_add instead of
// rebuilding descriptors.
struct Descs {
    uint64_t k_km, v_km, q_km, o_km;  // K-major (S^T, dP^T operands)
    uint64_t k_mn, s_mn, q_mn, o_mn;  // MN-major (dQ^T, dK, dV operands)
};
__device__ __forceinline__ Descs make_descs(uint32_t sbase) {
    Descs d;
    d.k_km = tc::sdesc_sw128(sbase + SM_K, 16, 1024);
    d.v_km = tc::sdesc_sw128(sbase + SM_V, 16, 1024);
    d.q_km = tc::sdesc_sw128(sbase + SM_Q, 16, 1024);
    d.o_km = tc::sdesc_sw128(sbase + SM_O, 16, 1024);
    d.k_mn = tc::sdesc_sw128(sbase + SM_K, kKV / 2, 1024);
    d.s_mn = tc::sdesc_sw128(sbase + SM_S, kKV / 2, 1024);
    d.q_mn = tc::sdesc_sw128(sbase + SM_Q, kQT / 2, 1024);
    d.o_mn = tc::sdesc_sw128(sbase + SM_O, kQT / 2, 1024);
    return d;
}
__device__ __forceinline__ uint64_t at(uint64_t desc, uint32_t bytes) { return tc::sdesc_add(desc, bytes); }

__device__ __forceinline__ bool issue_dq(const Descs& dd, const uint64_t* bar, uint32_t tmem, uint32_t ts, int s,
                                         volatile int* abort) {
    constexpr uint32_t id_dq = tc::idesc_bf16(D, BQ, 1) | (1u << 15);  // A and B MN-major
    // dQ^T of the previous step must have been read out of TMEM, and this
    // step's dS^T must be in shared memory (one barrier per step parity: the
    // P/dS warps cannot get two steps ahead, the step after next needs a
    // dP^T that is issued after this dQ^T)
    if (s >= 1 && !mma_wait(bar, B_DQF, (ts - 1) & 1, abort)) return false;
    if (!mma_wait(bar, B_SS + (ts & 1), (ts >> 1) & 1, abort)) return false;
    const uint64_t sS = at(dd.s_mn, (ts & 1) * kST);
#pragma unroll
    for (int k = 0; k < BN / 16; ++k) tc::mma_ss(tmem + TDQ, at(dd.k_mn, 2048 * k), at(sS, 2048 * k), id_dq, k > 0);
    tc::mma_commit(tc::smem_addr(&bar[B_DQ]));
    return true;
}

// S^T = K Q^T and dP^T = V dO^T of global step ts, once its Q and dO are in shared memory.
__device__ __forceinline__ bool issue_sdp(const Descs& dd, const uint64_t* bar, uint32_t tmem, uint32_t ts,
                                          volatile int* abort) {
    constexpr uint32_t id_st = tc::idesc_bf16(BN, BQ, 0);  // A, B K-major
    const uint32_t st = ts % kStages;
    if (!mma_wait(bar, B_QDF + st, (ts / kStages) & 1, abort)) return false;
    const uint64_t q = at(dd.q_km, st * kQT), o = at(dd.o_km, st * kQT);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
        const uint32_t oa = (k >> 2) * (kKV / 2) + (k & 3) * 32, ob = (k >> 2) * (kQT / 2) + (k & 3) * 32;
        tc::mma_ss(tmem + TS, at(dd.k_km, oa), at(q, ob), id_st, k > 0);
    }
    tc::mma_commit(tc::smem_addr(&bar[B_S]));
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
        const uint32_t oa = (k >> 2) * (kKV / 2) + (k & 3) * 32, ob = (k >> 2) * (kQT / 2) + (k & 3) * 32;
        tc::mma_ss(tmem + TDP, at(dd.v_km, oa), at(o, ob), id_st, k > 0);
    }
    tc::mma_commit(tc::smem_addr(&bar[B_DP]));
    return true;
}

// Per step s the tensor pipe receives S^T(s+1), dP^T(s+1), dV(s), dK(s),
// dQ^T(s): the next step's S^T and dP^T go in as soon as the P/dS warps have
// read S^T(s) and dP^T(s) into registers (B_LD), so they run while P/dS(s) is
// still computing; dV(s) and dK(s) wait for P^T(s) and dS^T(s) (B_SM).
__device__ __forceinline__ void issue_item(const ItemCtx& c, uint32_t sbase, const uint64_t* bar, uint32_t tmem,
                                           uint32_t ts_base, uint32_t item_count, volatile int* abort) {
    constexpr uint32_t id_kv = tc::idesc_bf16(BN, D, 1);  // dV, dK: A K-major (TMEM), B MN-major
    if (!mma_wait(bar, B_KV, item_count & 1, abort)) return;
    if (c.n_steps == 0) return;
    const Descs dd = make_descs(sbase);
    if (!issue_sdp(dd, bar, tmem, ts_base, abort)) return;
    for (int s = 0; s < c.n_steps; ++s) {
        const uint32_t ts = ts_base + s, st = ts % kStages;
        if (s + 1 < c.n_steps) {
            if (!mma_wait(bar, B_LD, ts & 1, abort)) return;
            if (!issue_sdp(dd, bar, tmem, ts + 1, abort)) return;
        }
        if (!mma_wait(bar, B_SM, ts & 1, abort)) return;
        // dV += P^T dO, dK += dS^T Q (P^T and dS^T in TMEM)
        const uint64_t q = at(dd.q_mn, st * kQT), o = at(dd.o_mn, st * kQT);
#pragma unroll
        for (int k = 0; k < BQ / 16; ++k)
            tc::mma_ts(tmem + TDV, tmem + TP + 8 * k, at(o, 2048 * k), id_kv, (s > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < BQ / 16; ++k)
            tc::mma_ts(tmem + TDK, tmem + TDS + 8 * k, at(q, 2048 * k), id_kv, (s > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(tc::smem_addr(&bar[B_QDE + st]));
        if (!issue_dq(dd, bar, tmem, ts, s, abort)) return;
    }
}

// ------------------------------------------------------------ P/dS group
// Thread = one key row (TMEM lane) x query columns 32g .. 32g + 31.
__device__ __forceinline__ void pds_item(const ItemCtx& c, const BwdArgs& a, uint8_t* smem, const uint64_t* bar,
                                         const StepInfo* info, uint32_t tmem, uint32_t ts_base, volatile int* abort) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp >> 2;
    const int kk = 32 * (warp & 3) + lane;  // key row in the tile == TMEM lane
    const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
    const float sl2 = a.scale_log2;
    // Row positions that see this thread's key, one interval per query range:
    // a clean key of block b is seen by clean rows of blocks >= b and corrupted
    // rows of blocks > b; a corrupted key only by the corrupted rows of its block.
    const KeyRows kr = key_rows(a.lay, c.kt, kk);
    int rem = 0;  // step index within the current query head
    for (int s = 0; s < c.n_steps; ++s) {
        const uint32_t ts = ts_base + s, st = ts % kStages;
        const bool in_a = rem < c.na;
        const int p0 = in_a ? c.ra_lo + rem * BQ : c.rb_lo + (rem - c.na) * BQ;
        const int nrows = imin(BQ, (in_a ? c.ra_hi : c.rb_hi) - p0);
        if (++rem == c.per_head) rem = 0;
        const int lo = imax((in_a ? kr.a_lo : kr.b_lo) - p0, 0) - 32 * g;  // relative to this group's first column
        const int hi = imin((in_a ? kr.a_hi : kr.b_hi) - p0, nrows) - 32 * g;
        const int len = imax(hi - lo, 0);
        const bool all_visible = __all_sync(0xffffffffu, lo <= 0 && hi >= 32);
        bool got = tc::mbar_wait(tc::smem_addr(&bar[B_QDF + st]), (ts / kStages) & 1, abort, kTimeoutNs);
        got = got && tc::mbar_wait(tc::smem_addr(&bar[B_S]), ts & 1, abort, kTimeoutNs);
        got = got && tc::mbar_wait(tc::smem_addr(&bar[B_DP]), ts & 1, abort, kTimeoutNs);
        if (!__all_sync(0xffffffffu, got)) return;
        tc::tc_fence_after();
        uint32_t sr[32], dr[32];
        tc::tmem_ld32(tmem + lb + TS + 32 * g, sr);
        tc::tmem_ld32(tmem + lb + TDP + 32 * g, dr);
        const float4* lse4 = reinterpret_cast<const float4*>(info[st].nl2 + 32 * g);
        const float4* ds4 = reinterpret_cast<const float4*>(info[st].dsum + 32 * g);
        tc::tmem_ld_wait();
        tc::tc_fence_before();
        tc::mbar_arrive(tc::smem_addr(&bar[B_LD]));  // S^T and dP^T of the next step may go
        uint32_t pp[16], dd[16];
        const float2 sl2x2 = make_float2(sl2, sl2);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 l4 = lse4[q], d4 = ds4[q];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int col = 4 * q + 2 * u;
                const float2 nl = u == 0 ? make_float2(l4.x, l4.y) : make_float2(l4.z, l4.w);
                const float2 dsum = u == 0 ? make_float2(d4.x, d4.y) : make_float2(d4.z, d4.w);
                const float2 x = tc::fma2(make_float2(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])), sl2x2, nl);
                float2 p = make_float2(ex2f(x.x), ex2f(x.y));
                if (!all_visible) {
                    p.x = (unsigned)(col - lo) < (unsigned)len ? p.x : 0.f;
                    p.y = (unsigned)(col + 1 - lo) < (unsigned)len ? p.y : 0.f;
                }
                const float2 ds = tc::mul2(p, tc::sub2(make_float2(__uint_as_float(dr[col]), __uint_as_float(dr[col + 1])), dsum));
                pp[2 * q + u] = pack2(p.x, p.y);
                dd[2 * q + u] = pack2(ds.x, ds.y);
            }
        }
        // P^T and dS^T of the previous step must have been read by its dV and dK
        if (ts > 0) {
            const uint32_t tp = ts - 1;
            got = tc::mbar_wait(tc::smem_addr(&bar[B_QDE + tp % kStages]), (tp / kStages) & 1, abort, kTimeoutNs);
            if (!__all_sync(0xffffffffu, got)) return;
            tc::tc_fence_after();
        }
        tc::tmem_st16(tmem + lb + TP + 16 * g, pp);
        tc::tmem_st16(tmem + lb + TDS + 16 * g, dd);
        tc::tmem_st_wait();
        tc::tc_fence_before();
        tc::mbar_arrive(tc::smem_addr(&bar[B_SM]));  // dV and dK may go
        {   // dS^T row kk, columns 32g..32g+31 = 16-byte chunks 4g..4g+3 of a 128-byte swizzled row
            uint8_t* srow = smem + SM_S + (ts & 1) * kST + kk * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int chunk = (4 * g + q) ^ (kk & 7);
                *reinterpret_cast<uint4*>(srow + chunk * 16) = make_uint4(dd[4 * q], dd[4 * q + 1], dd[4 * q + 2], dd[4 * q + 3]);
            }
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(tc::smem_addr(&bar[B_SS + (ts & 1)]));  // dQ^T may go (issued one step later)
    }
}

__device__ __forceinline__ void red_add_f32(float* p, float v) {
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// -------------------------------------------------------------- dq group
// Thread = one head-dim lane d of dQ^T (TMEM lane) x 64 query columns. With
// kRedDq the step's dq goes straight from registers into the fp32
// accumulator, one reduction per (row, d): a warp's 32 lanes cover 32
// consecutive d of one row, 128 contiguous bytes. Otherwise it goes out as two
// TMA reduce-adds of 32 rows through two staging buffers in shared memory.
// At the end of the item it writes dK and dV (thread = key row).
template <bool kRedDq>
__device__ __forceinline__ bool dq_item(const ItemCtx& c, const BwdArgs& a, uint32_t sbase, uint8_t* smem,
                                        const uint64_t* bar, uint32_t tmem, const CUtensorMap* tdq, uint32_t ts_base,
                                        volatile int* abort) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dl = 32 * (warp & 3) + lane;  // d index == TMEM lane
    const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
    const bool leader = tid == 256;
    if constexpr (kRedDq) {
        const long long rstride = (long long)a.H * D;
        for (int s = 0; s < c.n_steps; ++s) {
            const uint32_t ts = ts_base + s;
            const bool got = tc::mbar_wait(tc::smem_addr(&bar[B_DQ]), ts & 1, abort, kTimeoutNs);
            if (!__all_sync(0xffffffffu, got)) return false;
            tc::tc_fence_after();
            int h, p0, nrows;
            step_rows(c, a, s, &h, &p0, &nrows);
            uint32_t qv[2][32];
            tc::tmem_ld32(tmem + lb + TDQ, qv[0]);
            tc::tmem_ld32(tmem + lb + TDQ + 32, qv[1]);
            tc::tmem_ld_wait();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_addr(&bar[B_DQF]));  // dQ^T of the next step may go
            float* dst = a.dqacc + (long long)q_row_of(a.lay, c.kt, p0) * rstride + (long long)h * D + dl;
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (e < nrows) red_add_f32(dst + e * rstride, __uint_as_float(qv[0][e]));  // scaled in the convert kernel
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (32 + e < nrows) red_add_f32(dst + (32 + e) * rstride, __uint_as_float(qv[1][e]));
        }
    } else
    for (int s = 0; s < c.n_steps; ++s) {
        const uint32_t ts = ts_base + s;
        const bool got = tc::mbar_wait(tc::smem_addr(&bar[B_DQ]), ts & 1, abort, kTimeoutNs);
        if (!named_and(2, 128, got)) return false;
        tc::tc_fence_after();
        int h, p0, nrows;
        step_rows(c, a, s, &h, &p0, &nrows);
        uint32_t qv[2][32];
        tc::tmem_ld32(tmem + lb + TDQ, qv[0]);
        tc::tmem_ld32(tmem + lb + TDQ + 32, qv[1]);
        tc::tmem_ld_wait();
        tc::tc_fence_before();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            // staging buffer `half` was last read by the reduce issued one step ago
            if (leader) bulk_wait_read1();
            named_sync(2, 128);
            float* stg = reinterpret_cast<float*>(smem + SM_STG + half * kStg) + dl;
#pragma unroll
            for (int e = 0; e < 32; ++e) stg[e * D] = __uint_as_float(qv[half][e]);  // scaled in the convert kernel
            tc::fence_proxy_async_smem();
            named_sync(2, 128);
            if (leader) {
                tma_reduce_add_3d(tdq, sbase + SM_STG + half * kStg, 0, h, q_row_of(a.lay, c.kt, p0) + kHalfRows * half);
                bulk_commit();
                if (half == 1) tc::mbar_arrive(tc::smem_addr(&bar[B_DQF]));
            }
        }
    }
    // dK and dV: the last dQ^T commit covered every MMA of the item. Keys that
    // no query row of the call sees (clean keys after a block group's last
    // block) get zeros; their TMEM columns were never written for this item.
    const int kk = dl;
    const bool key_ok = kk < c.kv_rows;
    const bool seen = c.n_steps > 0;
    // dk, dv [slots, Lk, Hk, D]: a task list's tile writes its task's slot
    const int slot = a.lay.mode == MODE_TASKS ? ld_ro(&a.lay.tasks[c.kt.task].slot) : 0;
    const long long rowoff = ((long long)slot * a.Lk + c.k0 + kk) * ((long long)a.Hk * D) + (long long)c.kvh * D;
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
        const uint32_t src = which == 0 ? TDK : TDV;
        __nv_bfloat16* dst = (which == 0 ? a.dk : a.dv) + rowoff;
        const float mul = which == 0 ? a.scale : 1.f;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
            uint32_t v[32];
            if (seen) {
                tc::tmem_ld32(tmem + lb + src + 32 * q, v);
                tc::tmem_ld_wait();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
            if (key_ok) {
                uint4* o = reinterpret_cast<uint4*>(dst + 32 * q);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[e] = make_uint4(pack2(__uint_as_float(v[8 * e]) * mul, __uint_as_float(v[8 * e + 1]) * mul),
                                      pack2(__uint_as_float(v[8 * e + 2]) * mul, __uint_as_float(v[8 * e + 3]) * mul),
                                      pack2(__uint_as_float(v[8 * e + 4]) * mul, __uint_as_float(v[8 * e + 5]) * mul),
                                      pack2(__uint_as_float(v[8 * e + 6]) * mul, __uint_as_float(v[8 * e + 7]) * mul));
            }
        }
    }
    return true;
}

// ------------------------------------------------------------------ kernel
template <bool kRedDq>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc64_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = tc::smem_addr(smem);
    __shared__ __align__(8) uint64_t bar[B_COUNT];
    __shared__ __align__(16) StepInfo info[kStages];
    __shared__ uint32_t s_tmem;
    __shared__ int s_item;
    __shared__ int s_abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        s_abort = 0;
        tc::mbar_init(tc::smem_addr(&bar[B_KV]), 1);
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(tc::smem_addr(&bar[B_QDF + s]), 32);  // the loader's 32 lanes, after their stores
            tc::mbar_init(tc::smem_addr(&bar[B_QDE + s]), 1);
        }
        tc::mbar_init(tc::smem_addr(&bar[B_S]), 1);
        tc::mbar_init(tc::smem_addr(&bar[B_DP]), 1);
        tc::mbar_init(tc::smem_addr(&bar[B_SM]), 256);
        tc::mbar_init(tc::smem_addr(&bar[B_SS]), 256);
        tc::mbar_init(tc::smem_addr(&bar[B_SS + 1]), 256);
        tc::mbar_init(tc::smem_addr(&bar[B_DQ]), 1);
        tc::mbar_init(tc::smem_addr(&bar[B_DQF]), kRedDq ? 4 : 1);  // the dq warps' lane 0 / the TMA leader
        tc::mbar_init(tc::smem_addr(&bar[B_LD]), 256);
        tc::fence_barrier_init();
    }
    if (warp == 13) {
        tc::tmem_alloc(tc::smem_addr(&s_tmem), kTmemCols);
        tc::tmem_relinquish();
    }
    if (warp == 12 && lane == 0) {
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_do);
        tc::prefetch_tmap(&tm_dq);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* abort = &s_abort;
    const int n_items = a.hdr->n_tiles * a.Hk;
    uint32_t ts_base = 0, item_count = 0;
    for (;;) {
        __syncthreads();
        if (tid == 0) s_item = *abort ? n_items : atomicAdd(&a.hdr->counter, 1);
        __syncthreads();
        const int item = s_item;
        if (item >= n_items) break;
        const ItemCtx c = decode(a, item);
        if (warp == 12) {
            load_item(c, a, sbase, bar, info, &tm_k, &tm_v, &tm_q, &tm_do, ts_base, abort);
        } else if (warp == 13) {
            if (lane == 0) issue_item(c, sbase, bar, tmem, ts_base, item_count, abort);
        } else if (warp < 8) {
            pds_item(c, a, smem, bar, info, tmem, ts_base, abort);
        } else {
            dq_item<kRedDq>(c, a, sbase, smem, bar, tmem, &tm_dq, ts_base, abort);
        }
        ts_base += c.n_steps;
        ++item_count;
    }
    if (tid == 256) bulk_wait0();  // every dq reduce has landed
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 13) {
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

// [rows, heads, D] tensor as a 3-D map (D, heads, rows) with (box_d, 1, box_rows) boxes.
bool make_map(CUtensorMap* m, const void* base, bool f32, int heads, long long rows, int box_d, int box_rows,
              CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int esz = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * esz, (cuuint64_t)heads * D * esz};
    cuuint32_t box[3] = {(cuuint32_t)box_d, 1, (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_bwd_tc64_main(const BwdArgs& a, int num_sms, cudaStream_t st) {
    CUtensorMap mk, mv, mq, mdo, mdq;
    if (!make_map(&mk, a.k, false, a.Hk, a.Lk, 64, BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mv, a.v, false, a.Hk, a.Lk, 64, BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mq, a.q, false, a.H, a.Lq, 64, BQ, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mdo, a.dO, false, a.H, a.Lq, 64, BQ, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mdq, a.dqacc, true, a.H, a.Lq, D, kHalfRows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const char* mode = getenv("BDLM_BWD_DQ");
    const bool red = mode && mode[0] == 'r';
    auto kern = red ? bwd_tc64_kernel<true> : bwd_tc64_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<num_sms, kThreads, kSmemBytes, st>>>(mk, mv, mq, mdo, mdq, a);
    return cudaGetLastError();
}

}  // namespace bdlm
