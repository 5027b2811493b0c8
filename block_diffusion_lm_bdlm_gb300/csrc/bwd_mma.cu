// bwd_mma.cu - BDLM attention backward: preprocess and dq-convert kernels,
// and the warp-level tensor-core (mma.sync) main kernel used for head_dim 64
// (head_dim 128 runs the tcgen05 main kernel of bwd_tc.cu).
//
// Three kernels after the tile prologue:
//   1. preprocess: D_i = sum_d dO_i * o_i (fp32) per (row, head), and zero the
//      fp32 dq accumulator in the same pass;
//   2. main, key-major: one work item = (64-key tile, kv head). It loops over
//      the G query heads of the kv head and over the 64-row query tiles that
//      see the key tile (a clean key tile is seen by the clean rows from its
//      block on and by the corrupted rows of later blocks; a corrupted key tile
//      only by its own blocks' corrupted rows). Per step it recomputes
//      S^T = K Q^T, P^T = exp(S^T - lse), dP^T = V dO^T, dS^T = P^T (dP^T - D),
//      accumulates dV += P^T dO and dK += dS^T Q in registers (no atomics:
//      the item owns its keys for all G heads), and adds dq += dS K into the
//      fp32 accumulator with vector atomics;
//   3. convert: dq = bf16(accumulator), times the softmax scale when the
//      main kernel accumulated dS K unscaled (the tensor-core kernel).
#include <climits>
#include <cstdlib>

#include "common.cuh"
#include "kernels.h"
#include "warp_mma.cuh"

namespace bdlm {
namespace {

constexpr int BN = kBwdKeyTile;  // keys per item, 16 per warp
constexpr int BQ = kBwdQTile;    // query rows per step
constexpr int NT = 128;

template <int D>
constexpr int bwd_smem_bytes() {
    return 2 * BN * D * 2 + 4 * BQ * D * 2 + BN * BQ * 2;  // K, V, 2x(Q, dO), dS^T
}

// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdArgs a) {
    constexpr int LPR = D / 8;  // lanes per (row, head)
    const long long pair = ((long long)blockIdx.x * 256 + threadIdx.x) / LPR;
    const int c = threadIdx.x % LPR;
    const long long n_pairs = a.Lq * a.H;
    const bool ok = pair < n_pairs;  // whole lane groups are in or out
    const long long row = ok ? pair / a.H : 0;
    const int h = ok ? (int)(pair % a.H) : 0;
    const long long off = (ok ? pair : 0) * D + c * 8;
    float s = 0.f;
    if (ok) {
        const uint4 x = *reinterpret_cast<const uint4*>(a.dO + off);
        const uint4 y = *reinterpret_cast<const uint4*>(a.o + off);
        const uint32_t ux[4] = {x.x, x.y, x.z, x.w}, uy[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s = fmaf(__uint_as_float(ux[i] << 16), __uint_as_float(uy[i] << 16), s);
            s = fmaf(__uint_as_float(ux[i] & 0xffff0000u), __uint_as_float(uy[i] & 0xffff0000u), s);
        }
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o, LPR);
    if (!ok) return;
    if (c == 0) a.Dsum[(long long)h * a.Lq + row] = s;
    float4* acc = reinterpret_cast<float4*>(a.dqacc + off);
    acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
}

template <int D>
// dq = bf16(mul * accumulator): the tensor-core main kernel accumulates
// dS K unscaled (mul = softmax scale), the warp-level one scaled (mul = 1).
__global__ void __launch_bounds__(256) bwd_convert_kernel(const BwdArgs a, float mul) {
    const long long i = (long long)blockIdx.x * 256 + threadIdx.x;  // 8 elements each
    const long long n = a.Lq * a.H * D / 8;
    if (i >= n) return;
    const float4 x = reinterpret_cast<const float4*>(a.dqacc)[2 * i];
    const float4 y = reinterpret_cast<const float4*>(a.dqacc)[2 * i + 1];
    uint4 out;
    out.x = pack_bf16(x.x * mul, x.y * mul);
    out.y = pack_bf16(x.z * mul, x.w * mul);
    out.z = pack_bf16(y.x * mul, y.y * mul);
    out.w = pack_bf16(y.z * mul, y.w * mul);
    reinterpret_cast<uint4*>(a.dq)[i] = out;
}

// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(NT, 2) bwd_mma_kernel(const BwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sK = smem_u32(smem);
    const uint32_t sV = sK + BN * D * 2;
    const uint32_t sQ0 = sV + BN * D * 2;        // 2 buffers
    const uint32_t sO0 = sQ0 + 2 * BQ * D * 2;   // dO, 2 buffers
    const uint32_t sS = sO0 + 2 * BQ * D * 2;    // dS^T [BN][BQ]
    uint8_t* const sS_ptr = smem + (sS - sK);
    __shared__ Span s_span[2][BQ];
    __shared__ float s_lse2[2][BQ];
    __shared__ float s_D[2][BQ];
    __shared__ int s_rowfull[2][BQ];
    __shared__ int s_item;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tq = lane & 3;
    const int H = a.H, G = a.G;
    const int n_items = a.hdr->n_tiles * a.Hk;
    const long long q_stride = (long long)H * D;
    const long long k_stride = (long long)a.Hk * D;
    const float sl2 = a.scale_log2;

    for (;;) {
        if (tid == 0) s_item = atomicAdd(&a.hdr->counter, 1);
        __syncthreads();
        const int item = s_item;
        if (item >= n_items) break;
        const Tile kt = a.table[item / a.Hk];
        const int kvh = item % a.Hk;
        const int n = kt.n;
        const int k0 = key_row0(a.lay, kt);  // first k row of the item
        const int kv_rows = kt.nrows;

        // query ranges (row positions) that see these keys
        const KeyRows kr = key_tile_rows(a.lay, kt);
        const int ra_lo = kr.a_lo, ra_hi = kr.a_hi, rb_lo = kr.b_lo, rb_hi = kr.b_hi;
        const int na = (ra_hi - ra_lo + BQ - 1) / BQ;
        const int nb = (rb_hi - rb_lo + BQ - 1) / BQ;
        const int per_head = na + nb;
        const int n_steps = per_head * G;

        load_tile_async<D, BN, NT>(sK, a.k, k0, (long long)k0 + kv_rows, k_stride, kvh);
        load_tile_async<D, BN, NT>(sV, a.v, k0, (long long)k0 + kv_rows, k_stride, kvh);
        cp_async_commit();

        auto prefetch = [&](int s, int buf) {
            const int hh = s / per_head, rem = s % per_head;
            const int h = kvh * G + hh;
            const int p0 = rem < na ? ra_lo + rem * BQ : rb_lo + (rem - na) * BQ;
            const int hi = rem < na ? ra_hi : rb_hi;
            const Tile qt{kt.doc_start, n, p0, imin(BQ, hi - p0), kt.task};
            const long long qr0 = q_row_of(a.lay, kt, p0);
            load_tile_async<D, BQ, NT>(sQ0 + buf * BQ * D * 2, a.q, qr0, qr0 + qt.nrows, q_stride, h);
            load_tile_async<D, BQ, NT>(sO0 + buf * BQ * D * 2, a.dO, qr0, qr0 + qt.nrows, q_stride, h);
            cp_async_commit();
            if (tid < BQ) {
                const Span sp = row_span(a.lay, qt, tid);
                s_span[buf][tid] = sp;
                float l2 = INFINITY, dd = 0.f;
                if (tid < qt.nrows) {
                    const float lse = a.lse[(long long)h * a.Lq + qr0 + tid];
                    l2 = lse == -INFINITY ? INFINITY : lse * 1.4426950408889634f;
                    dd = a.Dsum[(long long)h * a.Lq + qr0 + tid];
                }
                s_lse2[buf][tid] = l2;
                s_D[buf][tid] = dd;
                s_rowfull[buf][tid] = tid < qt.nrows && kv_rows == BN && sp.p_lo <= k0 && k0 + BN <= sp.p_hi;
            }
        };

        float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = 0.f;
            dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;
        }

        if (n_steps > 0) prefetch(0, 0);
        for (int s = 0; s < n_steps; ++s) {
            const int buf = s & 1;
            if (s + 1 < n_steps) {
                prefetch(s + 1, buf ^ 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            const int full = __syncthreads_and(tid < BQ ? s_rowfull[buf][tid] : 1);
            const int hh = s / per_head, rem = s % per_head;
            const int h = kvh * G + hh;
            const int p0 = rem < na ? ra_lo + rem * BQ : rb_lo + (rem - na) * BQ;
            const int qrows = imin(BQ, (rem < na ? ra_hi : rb_hi) - p0);
            const long long qr0 = q_row_of(a.lay, kt, p0);
            const uint32_t sQ = sQ0 + buf * BQ * D * 2, sO = sO0 + buf * BQ * D * 2;

            // S^T and dP^T for this warp's 16 keys x 64 query rows
            float st[BQ / 8][4], dpt[BQ / 8][4];
#pragma unroll
            for (int i = 0; i < BQ / 8; ++i) {
                st[i][0] = st[i][1] = st[i][2] = st[i][3] = 0.f;
                dpt[i][0] = dpt[i][1] = dpt[i][2] = dpt[i][3] = 0.f;
            }
#pragma unroll
            for (int kc = 0; kc < D / 16; ++kc) {
                uint32_t ka[4], va[4];
                ldsm_x4(ka, sK + swz<D>(warp * 16 + (lane & 15), 2 * kc + (lane >> 4)));
                ldsm_x4(va, sV + swz<D>(warp * 16 + (lane & 15), 2 * kc + (lane >> 4)));
#pragma unroll
                for (int p = 0; p < BQ / 16; ++p) {
                    uint32_t b[4];
                    ldsm_x4(b, sQ + swz<D>(16 * p + (lane >> 4) * 8 + (lane & 7), 2 * kc + ((lane >> 3) & 1)));
                    mma_bf16(st[2 * p], ka, b[0], b[1]);
                    mma_bf16(st[2 * p + 1], ka, b[2], b[3]);
                    ldsm_x4(b, sO + swz<D>(16 * p + (lane >> 4) * 8 + (lane & 7), 2 * kc + ((lane >> 3) & 1)));
                    mma_bf16(dpt[2 * p], va, b[0], b[1]);
                    mma_bf16(dpt[2 * p + 1], va, b[2], b[3]);
                }
            }
            // P^T and dS^T
#pragma unroll
            for (int nt = 0; nt < BQ / 8; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int qc = nt * 8 + 2 * tq + (e & 1);
                    const int kk = warp * 16 + g + 8 * (e >> 1);
                    float p = fast_exp2(fmaf(st[nt][e], sl2, -s_lse2[buf][qc]));
                    if (!full) {
                        if (!(kk < kv_rows && span_sees(s_span[buf][qc], k0 + kk))) p = 0.f;
                    }
                    st[nt][e] = p;
                    dpt[nt][e] = p * (dpt[nt][e] - s_D[buf][qc]);
                }
            }
            // dV += P^T dO, dK += dS^T Q; stash dS^T for dq
#pragma unroll
            for (int kc = 0; kc < BQ / 16; ++kc) {
                uint32_t pa[4], da[4];
                pa[0] = pack_bf16(st[2 * kc][0], st[2 * kc][1]);
                pa[1] = pack_bf16(st[2 * kc][2], st[2 * kc][3]);
                pa[2] = pack_bf16(st[2 * kc + 1][0], st[2 * kc + 1][1]);
                pa[3] = pack_bf16(st[2 * kc + 1][2], st[2 * kc + 1][3]);
                da[0] = pack_bf16(dpt[2 * kc][0], dpt[2 * kc][1]);
                da[1] = pack_bf16(dpt[2 * kc][2], dpt[2 * kc][3]);
                da[2] = pack_bf16(dpt[2 * kc + 1][0], dpt[2 * kc + 1][1]);
                da[3] = pack_bf16(dpt[2 * kc + 1][2], dpt[2 * kc + 1][3]);
                // dS^T rows (keys) 16w+g and 16w+g+8, columns (queries) of chunks 2kc, 2kc+1
                const int r0 = warp * 16 + g;
                *reinterpret_cast<uint32_t*>(sS_ptr + swz<BQ>(r0, 2 * kc) + 4 * tq) = da[0];
                *reinterpret_cast<uint32_t*>(sS_ptr + swz<BQ>(r0 + 8, 2 * kc) + 4 * tq) = da[1];
                *reinterpret_cast<uint32_t*>(sS_ptr + swz<BQ>(r0, 2 * kc + 1) + 4 * tq) = da[2];
                *reinterpret_cast<uint32_t*>(sS_ptr + swz<BQ>(r0 + 8, 2 * kc + 1) + 4 * tq) = da[3];
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    uint32_t b[4];
                    ldsm_x4_t(b, sO + swz<D>(16 * kc + ((lane >> 3) & 1) * 8 + (lane & 7), 2 * dp + (lane >> 4)));
                    mma_bf16(dv[2 * dp], pa, b[0], b[1]);
                    mma_bf16(dv[2 * dp + 1], pa, b[2], b[3]);
                    ldsm_x4_t(b, sQ + swz<D>(16 * kc + ((lane >> 3) & 1) * 8 + (lane & 7), 2 * dp + (lane >> 4)));
                    mma_bf16(dk[2 * dp], da, b[0], b[1]);
                    mma_bf16(dk[2 * dp + 1], da, b[2], b[3]);
                }
            }
            __syncthreads();
            // dq[16 rows of this warp, D] += scale * dS K
            {
                float dq[D / 8][4];
#pragma unroll
                for (int i = 0; i < D / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;
#pragma unroll
                for (int kc = 0; kc < BN / 16; ++kc) {
                    uint32_t aa[4];
                    ldsm_x4_t(aa, sS + swz<BQ>(16 * kc + ((lane >> 4) & 1) * 8 + (lane & 7), 2 * warp + ((lane >> 3) & 1)));
#pragma unroll
                    for (int dp = 0; dp < D / 16; ++dp) {
                        uint32_t b[4];
                        ldsm_x4_t(b, sK + swz<D>(16 * kc + ((lane >> 3) & 1) * 8 + (lane & 7), 2 * dp + (lane >> 4)));
                        mma_bf16(dq[2 * dp], aa, b[0], b[1]);
                        mma_bf16(dq[2 * dp + 1], aa, b[2], b[3]);
                    }
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int r = warp * 16 + g + 8 * i;
                    if (r < qrows) {
                        float* dst = a.dqacc + (qr0 + r) * q_stride + (long long)h * D + 2 * tq;
#pragma unroll
                        for (int dn = 0; dn < D / 8; ++dn)
                            atomicAdd(reinterpret_cast<float2*>(dst + dn * 8),
                                      make_float2(dq[dn][2 * i] * a.scale, dq[dn][2 * i + 1] * a.scale));
                    }
                }
            }
            __syncthreads();
        }
        cp_async_wait<0>();

        // write dK (scaled) and dV for this warp's keys (dk, dv [slots, Lk,
        // Hk, D]: a task list's tile writes its task's slot)
        const long long kslot = a.lay.mode == MODE_TASKS ? (long long)ld_ro(&a.lay.tasks[kt.task].slot) * a.Lk : 0;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int kk = warp * 16 + g + 8 * i;
            if (kk < kv_rows) {
                __nv_bfloat16* dkr = a.dk + (kslot + k0 + kk) * k_stride + (long long)kvh * D + 2 * tq;
                __nv_bfloat16* dvr = a.dv + (kslot + k0 + kk) * k_stride + (long long)kvh * D + 2 * tq;
#pragma unroll
                for (int dn = 0; dn < D / 8; ++dn) {
                    *reinterpret_cast<uint32_t*>(dkr + dn * 8) =
                        pack_bf16(dk[dn][2 * i] * a.scale, dk[dn][2 * i + 1] * a.scale);
                    *reinterpret_cast<uint32_t*>(dvr + dn * 8) = pack_bf16(dv[dn][2 * i], dv[dn][2 * i + 1]);
                }
            }
        }
        __syncthreads();
    }
}

template <int D>
cudaError_t launch_bwd_t(const BwdArgs& a, int num_sms, cudaStream_t st) {
    const long long pairs = a.Lq * a.H;
    const long long pre_threads = pairs * (D / 8);
    bwd_pre_kernel<D><<<(unsigned)((pre_threads + 255) / 256), 256, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const char* kv = getenv("BDLM_BWD_K");
    const bool old = kv && kv[0] == 'o';
    if (!old) {
        e = launch_bwd_tc_main(a, num_sms, st);  // tensor-core main kernel, 128-key tiles
    } else if constexpr (D == 128) {
        e = launch_bwd_tc64_main(a, num_sms, st);
    } else {
        constexpr int smem = bwd_smem_bytes<D>();
        e = cudaFuncSetAttribute(bwd_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        bwd_mma_kernel<D><<<num_sms * 2, NT, smem, st>>>(a);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    const long long cv = pairs * D / 8;
    bwd_convert_kernel<D><<<(unsigned)((cv + 255) / 256), 256, 0, st>>>(a, (!old || D == 128) ? a.scale : 1.f);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, int num_sms, cudaStream_t st, int* launches) {
    cudaError_t e = a.D == 128 ? launch_bwd_t<128>(a, num_sms, st) : launch_bwd_t<64>(a, num_sms, st);
    if (e == cudaSuccess) *launches += 3;
    return e;
}

}  // namespace bdlm
