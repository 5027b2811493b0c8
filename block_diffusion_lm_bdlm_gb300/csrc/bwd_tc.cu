// bwd_tc.cu - BDLM attention backward main kernel on the 5th-generation
// tensor cores (head_dim 64 and 128).
//
// Key-major: one work item = (128-key tile, kv head). The item loops over the
// G query heads of the kv head and, for each, over the 128-row query steps
// that see the key tile (a clean key tile is seen by the clean rows from its
// block on and by the corrupted rows of later blocks; a corrupted key tile
// only by its own blocks' corrupted rows). Per step, every product is a
// 128 x 128 tensor-core tile, the shape at which tcgen05.mma runs at its full
// rate (a 64-wide B operand costs more shared-memory reads than the MMA has
// cycles):
//   S^T  = K Q^T          (M 128 keys, N 128 rows, K = d)          -> RS
//   dP^T = V dO^T                                                   -> RP
//   P^T  = exp2(S^T*scale*log2e - lse*log2e)   (compute warps; bf16 P^T
//          written over the S^T columns it came from)
//   dS^T = P^T (dP^T - D)  (bf16, over the dP^T columns, and to shared memory)
//   dV  += P^T dO         (A from TMEM)                             -> TMEM
//   dK  += dS^T Q         (A from TMEM)                             -> TMEM
//   d 128: dQ^T = K^T dS^T (M = d, N 128 rows, K 128 keys)           -> RP
//   d 64:  dQ   = dS K     (M 128 rows, N = d, K 128 keys)           -> own columns
//          read out and added into the fp32 dq accumulator from registers
//          (unscaled; the convert kernel applies the softmax scale).
// dK and dV stay in TMEM for the whole item (no atomics: the item owns its
// keys for all G heads) and are written once, as bf16, at the end.
//
// TMEM (512 columns): dK [0, d) | dV [d, 2d) | (d 64: dQ [128, 192)) |
// RS [256, 384) | RP [384, 512). The tensor pipe runs one CTA's MMAs in issue
// order, so an MMA may overwrite columns that an earlier-issued MMA reads:
// S^T(s+1) goes into RS right after dV(s) (which reads P^T(s) there), and for
// d 128 dQ^T(s) goes into RP right after dK(s) (which reads dS^T(s) there).
// Per step s the tensor pipe receives, in this order:
//   dP^T(s)  [RP free: dQ^T(s-1) read out]
//   dV(s)    [P^T(s) stored]
//   S^T(s+1) [Q(s+1) loaded]
//   dK(s)    [dS^T(s) stored]
//   dQ(s)    [d 64: dQ(s-1) read out]
// so that the compute warps work on P(s+1) while dK(s) and dQ(s) run, and on
// dS(s) while dV(s) and S^T(s+1) run.
//
// Warp roles (512 threads):
//   warps 0-7   P/dS groups: one TMEM lane = one key row; group g (warps
//               4g..4g+3) takes query columns 64g..64g+63 of a step. The mask
//               is analytic: for one key, the rows of a step that see it form
//               one interval (later clean blocks / later corrupted blocks for a
//               clean key, its own corrupted block for a corrupted key).
//               Group g writes its bf16 P^T and dS^T halves into its own
//               fp32 columns (RS / RP + 64g), so neither group overwrites
//               columns the other has not read yet.
//   warps 8-11  dq group: reads dQ^T (d 128: lane = d) or dQ (d 64: lane =
//               row) out of TMEM and reduces it into the fp32 dq accumulator;
//               writes dK and dV at the end of an item
//   warp  12    loader: TMA for K, V, Q, dO; plain loads for lse and D; two
//               stages for the per-step inputs
//   warp  13    TMEM owner and MMA issuer (one thread)
//   warps 14-15 idle: they complete the loader/MMA warpgroup, whose
//               registers setmaxnreg hands to the other roles
// Every mbarrier wait is bounded (2 s).
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace bdlm {
namespace {

constexpr int BN = 128;  // keys per item
constexpr int BQ = 128;  // query rows per step
constexpr int kThreads = 512;
constexpr int kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kStages = 2;

constexpr uint32_t TRS = 256, TRP = 384;

// Registers per thread: the launch gives every warp 128 (16 warps, 4 on each
// SM sub-partition of 512 per lane). setmaxnreg moves them between whole
// warpgroups: the loader/MMA warpgroup (warps 12-15, two of them idle) gives
// half of its share to the P/dS warpgroups and to the dq warpgroup, which
// holds a whole step of dQ^T (128 values) while it reduces it:
// 8 x 144 + 4 x 160 + 4 x 64 = 16 x 128, and per sub-partition (warps w,
// w+4, w+8, w+12) 144 + 144 + 160 + 64 = 512.
constexpr int kRegsPds = 144;
constexpr int kRegsDq = 160;
constexpr int kRegsIo = 64;

enum : int {
    B_KV = 0, B_QF = 1 /* x2 */, B_QE = 3 /* x2 */, B_OF = 5 /* x2 */, B_OE = 7 /* x2 */, B_S = 9, B_DP = 10,
    B_P = 11, B_DS = 12, B_DSS = 13, B_DQ = 14, B_DQF = 15, B_SF = 16, B_COUNT = 17
};

struct StepInfo {
    float nl2[BQ];   // -lse * log2(e) of the step's rows (0 beyond the step; those rows are masked)
    float dsum[BQ];  // D = rowsum(dO * o)
};

// Shared memory (offsets from a 1024-byte aligned base). Operand tiles are
// 128-byte swizzled [rows][64 columns] chunks of 16 KB.
template <int D>
struct Smem {
    static constexpr int kChunk = 128 * 128;           // [128 rows][64 bf16]
    static constexpr int kKV = BN * D * 2;             // K or V tile: D / 64 chunks
    static constexpr int kQT = BQ * D * 2;             // Q or dO tile: D / 64 chunks
    static constexpr int kST = BN * BQ * 2;            // dS^T [128 keys][128 rows]: 2 chunks of 64 rows
    static constexpr int K = 0;
    static constexpr int V = K + kKV;
    static constexpr int Q = V + kKV;                  // + stage * kQT
    static constexpr int O = Q + kStages * kQT;        // + stage * kQT
    static constexpr int S = O + kStages * kQT;
    static constexpr int INFO = S + kST;               // StepInfo[kStages]
    static constexpr int BAR = INFO + kStages * (int)sizeof(StepInfo);
    static constexpr int MISC = BAR + B_COUNT * 8;     // TMEM address, item, abort flag
    static constexpr int kBytes = MISC + 16;
};
static_assert(Smem<128>::kBytes <= 227 * 1024, "shared memory of the d 128 backward");

template <int D>
struct Tm {
    static constexpr uint32_t DK = 0, DV = D, DQ = 128;  // DQ: d 64 only
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
__device__ __forceinline__ void named_sync_all() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }
__device__ __forceinline__ void named_sync_dq() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
__device__ __forceinline__ void tma_reduce_add_3d(const void* tmap, uint32_t src, int c0, int c1, int c2) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(tmap),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void red_add_v4f32(float* p, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// Item -> (key tile, kv head). Tiles are ordered heaviest first. With many
// tiles (at least 8 per CTA) the items go in blocks of K = gridDim.x / 2
// tiles, kv head by kv head within a block, so one wave of gridDim.x items
// spans two kv heads: the CTAs running side by side then sweep the query rows
// of only those two kv heads' query heads, close together (neighbouring key
// tiles start their sweeps a tile apart), and their Q, dO tiles and the dq
// accumulator rows they add into are shared in L2. Measured on a GB300 at
// 128K + 128K rows, this took the backward from 808 to 542 ms (strictly
// heaviest first, one wave spans all kv heads and its sweeps outgrow L2).
// With fewer tiles (K = 1) the items of one tile (its kv heads) are
// consecutive and the order is strictly heaviest first.
__device__ __forceinline__ ItemCtx decode(const BwdArgs& a, int item) {
    ItemCtx c;
    const int nt = a.hdr->n_tiles;
    const int K = nt >= 8 * (int)gridDim.x ? (int)gridDim.x / 2 : 1;
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

// query rows of step s: head, first row position, valid rows
__device__ __forceinline__ void step_rows(const ItemCtx& c, const BwdArgs& a, int s, int* h, int* p0, int* nrows) {
    const int hh = s / c.per_head, rem = s % c.per_head;
    *h = c.kvh * a.G + hh;
    *p0 = rem < c.na ? c.ra_lo + rem * BQ : c.rb_lo + (rem - c.na) * BQ;
    const int hi = rem < c.na ? c.ra_hi : c.rb_hi;
    *nrows = imin(BQ, hi - *p0);
}

// The part of an item the dq warps need per step, kept in registers for the
// item: head, q row and valid rows of every step (q row = qbase + position).
struct StepMap {
    int h0, per_head, na, ra_lo, ra_hi, rb_lo, rb_hi, qbase;
    __device__ __forceinline__ StepMap(const ItemCtx& c, const BwdArgs& a)
        : h0(c.kvh * a.G), per_head(c.per_head), na(c.na), ra_lo(c.ra_lo), ra_hi(c.ra_hi), rb_lo(c.rb_lo),
          rb_hi(c.rb_hi), qbase(q_row_of(a.lay, c.kt, 0)) {}
    __device__ __forceinline__ void rows(int s, int* h, int* qrow, int* nrows) const {
        const int hh = s / per_head, rem = s % per_head;
        *h = h0 + hh;
        const int p0 = rem < na ? ra_lo + rem * BQ : rb_lo + (rem - na) * BQ;
        *nrows = imin(BQ, (rem < na ? ra_hi : rb_hi) - p0);
        *qrow = qbase + p0;
    }
};

// ---------------------------------------------------------------- loader
template <int D>
__device__ __forceinline__ void load_item(const ItemCtx& c, const BwdArgs& a, uint32_t sbase, const uint64_t* bar,
                                          StepInfo* info, const CUtensorMap* tk, const CUtensorMap* tv,
                                          const CUtensorMap* tq, const CUtensorMap* tdo, uint32_t ts_base,
                                          volatile int* abort) {
    using L = Smem<D>;
    constexpr int NC = D / 64;
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        const uint32_t bkv = tc::smem_addr(&bar[B_KV]);
        tc::mbar_arrive_expect_tx(bkv, 2 * L::kKV);
        for (int ch = 0; ch < NC; ++ch) {
            tc::tma_load_3d(sbase + L::K + ch * L::kChunk, tk, bkv, 64 * ch, c.kvh, c.k0);
            tc::tma_load_3d(sbase + L::V + ch * L::kChunk, tv, bkv, 64 * ch, c.kvh, c.k0);
        }
    }
    for (int s = 0; s < c.n_steps; ++s) {
        const uint32_t ts = ts_base + s, st = ts % kStages, ph = (ts / kStages) & 1;
        // Q stage (with the step's lse and D): free once dK two steps back
        // has read it. dO stage: for d 128, once the dq warps' staging of two
        // steps back has been reduced out of it; for d 64, with the Q stage.
        // Each tile goes as soon as its own stage is free.
        bool got = tc::mbar_wait(tc::smem_addr(&bar[B_QE + st]), ph ^ 1, abort, kTimeoutNs);
        if (!__all_sync(0xffffffffu, got)) return;
        int h, p0, nrows;
        step_rows(c, a, s, &h, &p0, &nrows);
        const int qr0 = q_row_of(a.lay, c.kt, p0);
        const uint32_t bf = tc::smem_addr(&bar[B_QF + st]);
        if (lane == 0) {
            mbar_expect_tx(bf, L::kQT);
            for (int ch = 0; ch < NC; ++ch)
                tc::tma_load_3d(sbase + L::Q + st * L::kQT + ch * L::kChunk, tq, bf, 64 * ch, h, qr0);
        }
        // lse and D: plain loads (the loader runs a step ahead of the MMAs),
        // stored pre-scaled so that P/dS spends one FFMA per element before exp2
        StepInfo& inf = info[st];
#pragma unroll
        for (int u = 0; u < BQ / 32; ++u) {
            const int r = (BQ / 32) * lane + u;
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
        if (D == 128) got = tc::mbar_wait(tc::smem_addr(&bar[B_OE + st]), ph ^ 1, abort, kTimeoutNs);
        if (!__all_sync(0xffffffffu, got)) return;
        if (lane == 0) {
            const uint32_t bo = tc::smem_addr(&bar[B_OF + st]);
            tc::mbar_arrive_expect_tx(bo, L::kQT);
            for (int ch = 0; ch < NC; ++ch)
                tc::tma_load_3d(sbase + L::O + st * L::kQT + ch * L::kChunk, tdo, bo, 64 * ch, h, qr0);
        }
    }
}

// ------------------------------------------------------------------- MMA
__device__ __forceinline__ bool mma_wait(const uint64_t* bar, int i, uint32_t parity, volatile int* abort) {
    if (!tc::mbar_wait(tc::smem_addr(&bar[i]), parity, abort, kTimeoutNs)) return false;
    tc::tc_fence_after();
    return true;
}

// Shared-memory descriptors of the operand tiles at stage 0; the MMA thread
// steps to K slices and stages with tc::sdesc_add.
template <int D>
struct Descs {
    uint64_t k_km, v_km, q_km, o_km;  // K-major (S^T, dP^T operands)
    uint64_t k_mn, s_mn, q_mn, o_mn;  // MN-major (dQ, dK, dV operands)
    __device__ __forceinline__ explicit Descs(uint32_t sbase) {
        using L = Smem<D>;
        k_km = tc::sdesc_sw128(sbase + L::K, 16, 1024);
        v_km = tc::sdesc_sw128(sbase + L::V, 16, 1024);
        q_km = tc::sdesc_sw128(sbase + L::Q, 16, 1024);
        o_km = tc::sdesc_sw128(sbase + L::O, 16, 1024);
        k_mn = tc::sdesc_sw128(sbase + L::K, L::kChunk, 1024);
        s_mn = tc::sdesc_sw128(sbase + L::S, L::kChunk, 1024);
        q_mn = tc::sdesc_sw128(sbase + L::Q, L::kChunk, 1024);
        o_mn = tc::sdesc_sw128(sbase + L::O, L::kChunk, 1024);
    }
};
__device__ __forceinline__ uint64_t at(uint64_t desc, uint32_t bytes) { return tc::sdesc_add(desc, bytes); }

// A[keys, K = d] x B[rows, K = d]^T into the 128 x 128 fp32 columns at dst
// (S^T from K and Q, dP^T from V and dO), both operands K-major.
template <int D>
__device__ __forceinline__ void mma_kq(uint32_t dst, uint64_t a, uint64_t b) {
    constexpr uint32_t id = tc::idesc_bf16(BN, BQ, 0);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * Smem<D>::kChunk + (k & 3) * 32;
        tc::mma_ss(dst, at(a, off), at(b, off), id, k > 0);
    }
}

// The columns of group g's K slices of a bf16 operand written over fp32
// columns (P^T over RS, dS^T over RP): slice k (rows 16k..16k+15 of the step)
// belongs to group k / 4 and sits at base + 64 (k / 4) + 8 (k % 4).
__device__ __forceinline__ uint32_t slice_col(int k) { return 64u * (uint32_t)(k >> 2) + 8u * (uint32_t)(k & 3); }

template <int D>
__device__ __forceinline__ void issue_item(const ItemCtx& c, uint32_t sbase, const uint64_t* bar, uint32_t tmem,
                                           uint32_t ts_base, uint32_t item_count, volatile int* abort) {
    using L = Smem<D>;
    using T = Tm<D>;
    constexpr uint32_t id_kv = tc::idesc_bf16(BN, D, 1);                 // dV, dK: A from TMEM, B MN-major
    constexpr uint32_t id_dq = D == 128 ? tc::idesc_bf16(D, BQ, 1) | (1u << 15)   // dQ^T: A, B MN-major
                                        : tc::idesc_bf16(BQ, D, 1) | (1u << 15);  // dQ:   A, B MN-major
    if (!mma_wait(bar, B_KV, item_count & 1, abort)) return;
    if (c.n_steps == 0) return;
    const Descs<D> dd(sbase);
    {   // S^T of the item's first step
        const uint32_t st = ts_base % kStages;
        if (!mma_wait(bar, B_QF + st, (ts_base / kStages) & 1, abort)) return;
        mma_kq<D>(tmem + TRS, dd.k_km, at(dd.q_km, st * L::kQT));
        tc::mma_commit(tc::smem_addr(&bar[B_S]));
    }
    for (int s = 0; s < c.n_steps; ++s) {
        const uint32_t ts = ts_base + s, st = ts % kStages;
        // dP^T(s) into RP (for d 128, RP last held dQ^T(s-1)), once dO(s) is in
        if (D == 128 && ts > 0 && !mma_wait(bar, B_DQF, (ts - 1) & 1, abort)) return;
        if (!mma_wait(bar, B_OF + st, (ts / kStages) & 1, abort)) return;
        mma_kq<D>(tmem + TRP, dd.v_km, at(dd.o_km, st * L::kQT));
        tc::mma_commit(tc::smem_addr(&bar[B_DP]));
        // dV += P^T dO
        if (!mma_wait(bar, B_P, ts & 1, abort)) return;
        const uint64_t o = at(dd.o_mn, st * L::kQT), q = at(dd.q_mn, st * L::kQT);
#pragma unroll
        for (int k = 0; k < BQ / 16; ++k)
            tc::mma_ts(tmem + T::DV, tmem + TRS + slice_col(k), at(o, 2048 * k), id_kv, (s > 0 || k > 0) ? 1u : 0u);
        // S^T(s+1) into RS (after dV(s) in the pipe, which read P^T(s) there)
        if (s + 1 < c.n_steps) {
            const uint32_t tn = ts + 1, sn = tn % kStages;
            if (!mma_wait(bar, B_QF + sn, (tn / kStages) & 1, abort)) return;
            mma_kq<D>(tmem + TRS, dd.k_km, at(dd.q_km, sn * L::kQT));
            tc::mma_commit(tc::smem_addr(&bar[B_S]));
        }
        // dK += dS^T Q
        if (!mma_wait(bar, B_DS, ts & 1, abort)) return;
#pragma unroll
        for (int k = 0; k < BQ / 16; ++k)
            tc::mma_ts(tmem + T::DK, tmem + TRP + slice_col(k), at(q, 2048 * k), id_kv, (s > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(tc::smem_addr(&bar[B_QE + st]));  // Q(s) (and dO(s)) read by every MMA that needs them
        // dq of this step from dS^T in shared memory and the K tile
        if (!mma_wait(bar, B_DSS, ts & 1, abort)) return;
        if (D == 128) {  // dQ^T = K^T dS^T into RP (after dK(s) in the pipe, which read dS^T(s) there)
#pragma unroll
            for (int k = 0; k < BN / 16; ++k)
                tc::mma_ss(tmem + TRP, at(dd.k_mn, 2048 * k), at(dd.s_mn, 2048 * k), id_dq, k > 0);
        } else {         // dQ = dS K into its own columns, once dQ(s-1) has been read out
            if (ts > 0 && !mma_wait(bar, B_DQF, (ts - 1) & 1, abort)) return;
#pragma unroll
            for (int k = 0; k < BN / 16; ++k)
                tc::mma_ss(tmem + T::DQ, at(dd.s_mn, 2048 * k), at(dd.k_mn, 2048 * k), id_dq, k > 0);
        }
        tc::mma_commit(tc::smem_addr(&bar[B_DQ]));
    }
}

// ------------------------------------------------------------ P/dS group
// Thread = one key row (TMEM lane) x query columns 64g .. 64g + 63.
template <int D>
__device__ __forceinline__ void pds_item(const ItemCtx& c, const BwdArgs& a, uint8_t* smem, const uint64_t* bar,
                                         const StepInfo* info, uint32_t tmem, uint32_t ts_base, volatile int* abort) {
    using L = Smem<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp >> 2;
    const int kk = 32 * (warp & 3) + lane;  // key row in the tile == TMEM lane
    const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lb + TRS + 64 * g, tP = tmem + lb + TRP + 64 * g;
    const float2 sl2x2 = make_float2(a.scale_log2, a.scale_log2);
    // Row positions that see this thread's key, one interval per query range:
    // a clean key of block b is seen by clean rows of blocks >= b and corrupted
    // rows of blocks > b; a corrupted key only by the corrupted rows of its block.
    const KeyRows kr = key_rows(a.lay, c.kt, kk);
    uint8_t* srow = smem + L::S + g * L::kChunk + kk * 128;  // this thread's row of dS^T, chunk g
    int rem = 0;  // step index within the current query head
    for (int s = 0; s < c.n_steps; ++s) {
        const uint32_t ts = ts_base + s, st = ts % kStages;
        const bool in_a = rem < c.na;
        const int p0 = in_a ? c.ra_lo + rem * BQ : c.rb_lo + (rem - c.na) * BQ;
        const int nrows = imin(BQ, (in_a ? c.ra_hi : c.rb_hi) - p0);
        if (++rem == c.per_head) rem = 0;
        const int lo = imax((in_a ? kr.a_lo : kr.b_lo) - p0, 0) - 64 * g;  // relative to this group's first column
        const int hi = imin((in_a ? kr.a_hi : kr.b_hi) - p0, nrows) - 64 * g;
        const int len = imax(hi - lo, 0);
        const bool all_visible = __all_sync(0xffffffffu, lo <= 0 && hi >= 64);
        // ---- P^T = exp2(S^T scale log2e - lse log2e), masked; bf16 over RS + 64g
        bool got = tc::mbar_wait(tc::smem_addr(&bar[B_QF + st]), (ts / kStages) & 1, abort, kTimeoutNs);
        got = got && tc::mbar_wait(tc::smem_addr(&bar[B_S]), ts & 1, abort, kTimeoutNs);
        if (!__all_sync(0xffffffffu, got)) return;
        tc::tc_fence_after();
        float p[64];
        {
            uint32_t r0[32], r1[32];
            tc::tmem_ld32(tS, r0);
            tc::tmem_ld32(tS + 32, r1);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                p[e] = __uint_as_float(r0[e]);
                p[32 + e] = __uint_as_float(r1[e]);
            }
        }
        const float4* nl4 = reinterpret_cast<const float4*>(info[st].nl2 + 64 * g);
        uint32_t pk[32];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float4 l4 = nl4[q];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int col = 4 * q + 2 * u;
                const float2 nl = u == 0 ? make_float2(l4.x, l4.y) : make_float2(l4.z, l4.w);
                const float2 x = tc::fma2(make_float2(p[col], p[col + 1]), sl2x2, nl);
                float2 e2 = make_float2(ex2f(x.x), ex2f(x.y));
                if (!all_visible) {
                    e2.x = (unsigned)(col - lo) < (unsigned)len ? e2.x : 0.f;
                    e2.y = (unsigned)(col + 1 - lo) < (unsigned)len ? e2.y : 0.f;
                }
                p[col] = e2.x;
                p[col + 1] = e2.y;
                pk[2 * q + u] = pack2(e2.x, e2.y);
            }
        }
        tc::tmem_st32(tS, pk);
        tc::tmem_st_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_addr(&bar[B_P]));  // dV(s) and then S^T(s+1) may go
        // ---- dS^T = P^T (dP^T - D), bf16 over RP + 64g (for dK), then into
        // shared memory (for dQ)
        got = tc::mbar_wait(tc::smem_addr(&bar[B_DP]), ts & 1, abort, kTimeoutNs);
        if (!__all_sync(0xffffffffu, got)) return;
        tc::tc_fence_after();
        const float4* ds4 = reinterpret_cast<const float4*>(info[st].dsum + 64 * g);
        uint32_t dk[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t r[32];
            tc::tmem_ld32(tP + 32 * half, r);
            tc::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 d4 = ds4[8 * half + q];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = 4 * q + 2 * u, col = 32 * half + e;
                    const float2 dsum = u == 0 ? make_float2(d4.x, d4.y) : make_float2(d4.z, d4.w);
                    const float2 ds = tc::mul2(make_float2(p[col], p[col + 1]),
                                               tc::sub2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), dsum));
                    dk[16 * half + 2 * q + u] = pack2(ds.x, ds.y);
                }
            }
        }
        tc::tmem_st32(tP, dk);
        tc::tmem_st_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_addr(&bar[B_DS]));  // dK(s) may go
        // the shared-memory dS^T buffer is free: d 128, the dq warps' staging
        // of step s-1 has been reduced out of it; d 64, dQ(s-1) has read it
        got = ts == 0 || tc::mbar_wait(tc::smem_addr(&bar[D == 128 ? B_SF : B_DQ]), (ts - 1) & 1, abort, kTimeoutNs);
        if (!__all_sync(0xffffffffu, got)) return;
        // row kk of dS^T chunk g: eight 16-byte units, 128-byte swizzled
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int unit = q ^ (kk & 7);
            *reinterpret_cast<uint4*>(srow + unit * 16) = make_uint4(dk[4 * q], dk[4 * q + 1], dk[4 * q + 2], dk[4 * q + 3]);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_addr(&bar[B_DSS]));  // dQ(s) may go
    }
}

// -------------------------------------------------------------- dq group
// d 128: thread = one head-dim lane d of dQ^T (TMEM lane) x the step's 128
// query columns; a warp's 32 lanes reduce 32 consecutive d of one row (128
// contiguous bytes) per instruction. d 64: thread = one query row of dQ x 64
// d; 16-byte vector reductions. At the end of the item it writes dK and dV
// (thread = key row).
// (The step loop keeps only the few values it needs live, from a decode at
// the start of the item; the item is decoded again for the dK, dV epilogue,
// which keeps the dq warps within their register budget while they hold a
// whole step of dQ^T.)
template <int D>
__device__ __forceinline__ bool dq_item(int item, int n_steps, const BwdArgs& a, uint8_t* smem, uint32_t sbase,
                                        const uint64_t* bar, uint32_t tmem, const CUtensorMap* tdq, uint32_t ts_base,
                                        volatile int* abort) {
    using T = Tm<D>;
    using L = Smem<D>;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dl = 32 * (warp & 3) + lane;  // TMEM lane
    const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
    const long long rstride = (long long)a.H * D;
    const StepMap sm(decode(a, item), a);
    for (int s = 0; s < n_steps; ++s) {
        const uint32_t ts = ts_base + s;
        int h, qrow, nrows;
        sm.rows(s, &h, &qrow, &nrows);
        const bool got = tc::mbar_wait(tc::smem_addr(&bar[B_DQ]), ts & 1, abort, kTimeoutNs);
        if (!__all_sync(0xffffffffu, got)) return false;
        tc::tc_fence_after();
        if constexpr (D == 128) {
            uint32_t v[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) tc::tmem_ld32(tmem + lb + TRP + 32 * q, v[q]);
            tc::tmem_ld_wait();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_addr(&bar[B_DQF]));  // RP may take dP^T(s+1)
            // Stage the step's dq as fp32 [64 rows][128 d] in two buffers that
            // are idle now (the dS^T buffer, read by dQ^T(s), and the dO(s)
            // stage, read by dP^T(s) and dV(s)), and add each into the fp32
            // accumulator with one TMA reduce-add. The dS^T buffer goes first
            // and is released as soon as its reduce has read it, since the
            // next step's dS^T waits for it. A warp writes 32 consecutive d
            // of one row per store.
            const uint32_t st = ts % kStages;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint32_t buf = half == 0 ? L::S : L::O + st * L::kQT;
                float* stg = reinterpret_cast<float*>(smem + buf) + dl;
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int e = 0; e < 32; ++e) stg[(32 * q + e) * D] = __uint_as_float(v[2 * half + q][e]);
                tc::fence_proxy_async_smem();
                named_sync_dq();
                if (dl == 0) {
                    if (64 * half < nrows) tma_reduce_add_3d(tdq, sbase + buf, 0, h, qrow + 64 * half);
                    bulk_commit();
                }
            }
            if (dl == 0) {
                bulk_wait_read1();  // the dS^T buffer has been read
                tc::mbar_arrive(tc::smem_addr(&bar[B_SF]));       // dS^T of the next step may be stored
                bulk_wait_read0();  // the dO(s) stage has been read
                tc::mbar_arrive(tc::smem_addr(&bar[B_OE + st]));  // dO of step s + 2 may be loaded
            }
        } else {
            uint32_t v[2][32];
            tc::tmem_ld32(tmem + lb + T::DQ, v[0]);
            tc::tmem_ld32(tmem + lb + T::DQ + 32, v[1]);
            tc::tmem_ld_wait();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_addr(&bar[B_DQF]));  // dQ(s+1) may go
            if (dl < nrows) {
                float* dst = a.dqacc + (long long)(qrow + dl) * rstride + (long long)h * D;
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        red_add_v4f32(dst + 32 * q + e, __uint_as_float(v[q][e]), __uint_as_float(v[q][e + 1]),
                                      __uint_as_float(v[q][e + 2]), __uint_as_float(v[q][e + 3]));
            }
        }
    }
    // dK and dV: the last dq commit covered every MMA of the item. Keys that
    // no query row of the call sees (clean keys after a block group's last
    // block) get zeros; their TMEM columns were never written for this item.
    const ItemCtx c = decode(a, item);
    const int kk = dl;
    const bool key_ok = kk < c.kv_rows;
    const bool seen = c.n_steps > 0;
    // dk, dv [slots, Lk, Hk, D]: a task list's tile writes its task's slot
    const int slot = a.lay.mode == MODE_TASKS ? ld_ro(&a.lay.tasks[c.kt.task].slot) : 0;
    const long long rowoff = ((long long)slot * a.Lk + c.k0 + kk) * ((long long)a.Hk * D) + (long long)c.kvh * D;
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
        const uint32_t src = which == 0 ? T::DK : T::DV;
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
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a) {
    using L = Smem<D>;
    // everything lives in dynamic shared memory, whose base the 128-byte
    // swizzled operand tiles need 1024-byte aligned
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = tc::smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (sbase & 1023u) {  // uniform over the CTA: nothing has been set up yet
        if (tid == 0) set_error(a.hdr, DEV_CHECK, -3);
        return;
    }
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR);
    StepInfo* info = reinterpret_cast<StepInfo*>(smem + L::INFO);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::MISC);
    int* s_item = reinterpret_cast<int*>(smem + L::MISC + 4);
    int* s_abort = reinterpret_cast<int*>(smem + L::MISC + 8);

    if (tid == 0) {
        *s_abort = 0;
        tc::mbar_init(tc::smem_addr(&bar[B_KV]), 1);
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(tc::smem_addr(&bar[B_QF + s]), 32);  // the loader's 32 lanes, after their stores
            tc::mbar_init(tc::smem_addr(&bar[B_QE + s]), 1);
            tc::mbar_init(tc::smem_addr(&bar[B_OF + s]), 1);  // the loader's lane 0 (+ the dO bytes)
            tc::mbar_init(tc::smem_addr(&bar[B_OE + s]), 1);  // the dq leader, after its reduce read the stage
        }
        tc::mbar_init(tc::smem_addr(&bar[B_S]), 1);
        tc::mbar_init(tc::smem_addr(&bar[B_DP]), 1);
        tc::mbar_init(tc::smem_addr(&bar[B_P]), 8);    // lane 0 of each P/dS warp, after its warp's stores
        tc::mbar_init(tc::smem_addr(&bar[B_DS]), 8);
        tc::mbar_init(tc::smem_addr(&bar[B_DSS]), 8);
        tc::mbar_init(tc::smem_addr(&bar[B_DQ]), 1);
        tc::mbar_init(tc::smem_addr(&bar[B_DQF]), 4);  // lane 0 of each dq warp
        tc::mbar_init(tc::smem_addr(&bar[B_SF]), 1);   // the dq leader
        tc::fence_barrier_init();
    }
    if (warp == 13) {
        tc::tmem_alloc(tc::smem_addr(s_tmem), kTmemCols);
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
    const uint32_t tmem = *s_tmem;
    volatile int* abort = s_abort;
    const int n_items = a.hdr->n_tiles * a.Hk;
    // Every role runs its own copy of the item loop (so that setmaxnreg can
    // give each role its register count); the loops meet at named barrier 1,
    // all 512 threads, twice per item.
    auto next_item = [&]() -> int {
        named_sync_all();
        if (tid == 0) *s_item = *abort ? n_items : atomicAdd(&a.hdr->counter, 1);
        named_sync_all();
        return *s_item;
    };
    uint32_t ts_base = 0, item_count = 0;
    if (warp >= 12) {
        tc::regs_dec<kRegsIo>();
        for (int item; (item = next_item()) < n_items;) {
            const ItemCtx c = decode(a, item);
            if (warp == 12)
                load_item<D>(c, a, sbase, bar, info, &tm_k, &tm_v, &tm_q, &tm_do, ts_base, abort);
            else if (warp == 13 && lane == 0)
                issue_item<D>(c, sbase, bar, tmem, ts_base, item_count, abort);
            // warps 14-15 only complete the warpgroup
            ts_base += c.n_steps;
            ++item_count;
        }
    } else if (warp >= 8) {
        tc::regs_inc<kRegsDq>();
        for (int item; (item = next_item()) < n_items;) {
            const int n_steps = decode(a, item).n_steps;
            dq_item<D>(item, n_steps, a, smem, sbase, bar, tmem, &tm_dq, ts_base, abort);
            ts_base += n_steps;
        }
    } else {
        tc::regs_inc<kRegsPds>();
        for (int item; (item = next_item()) < n_items;) {
            const ItemCtx c = decode(a, item);
            pds_item<D>(c, a, smem, bar, info, tmem, ts_base, abort);
            ts_base += c.n_steps;
        }
    }
    if (D == 128 && tid == 256) bulk_wait0();  // every dq reduce-add has landed
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && *s_abort) set_error(a.hdr, DEV_TIMEOUT, blockIdx.x);
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

// bf16 [rows, heads, d] tensor as a 3-D map (d, heads, rows) with 64 x 1 x
// box_rows boxes, 128-byte swizzled.
bool make_map(CUtensorMap* m, const void* base, int d, int heads, long long rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The fp32 dq accumulator [rows, heads, d] as a 3-D map (d, heads, rows) with
// d x 1 x 64 boxes, unswizzled: the target of the staged reduce-adds.
bool make_acc_map(CUtensorMap* m, float* base, int d, int heads, long long rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)heads * d * 4};
    cuuint32_t box[3] = {(cuuint32_t)d, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_t(const BwdArgs& a, int num_sms, cudaStream_t st) {
    CUtensorMap mk, mv, mq, mdo, mdq;
    if (!make_map(&mk, a.k, D, a.Hk, a.Lk, BN) || !make_map(&mv, a.v, D, a.Hk, a.Lk, BN) ||
        !make_map(&mq, a.q, D, a.H, a.Lq, BQ) || !make_map(&mdo, a.dO, D, a.H, a.Lq, BQ) ||
        !make_acc_map(&mdq, a.dqacc, D, a.H, a.Lq))
        return cudaErrorInvalidValue;
    constexpr int smem = Smem<D>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    bwd_tc_kernel<D><<<num_sms, kThreads, smem, st>>>(mk, mv, mq, mdo, mdq, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc_main(const BwdArgs& a, int num_sms, cudaStream_t st) {
    return a.D == 128 ? launch_t<128>(a, num_sms, st) : launch_t<64>(a, num_sms, st);
}

}  // namespace bdlm
