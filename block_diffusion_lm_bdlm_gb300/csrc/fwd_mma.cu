// fwd_mma.cu - BDLM attention forward on warp-level tensor cores
// (mma.sync m16n8k16 bf16 -> fp32), persistent over the ordered tile list.
//
// Per work item (64-row query tile, query head): the tile's rows iterate the
// union of their prefix intervals, then the union of their own-block
// intervals, 64 keys at a time, with K/V double-buffered through cp.async.
// Only tiles that are not fully visible to every row apply the element mask.
// Online softmax runs in base 2 in fp32 registers (row max and row sum via
// quad shuffles); lse is returned in natural-log units of the scaled logits.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "warp_mma.cuh"

namespace bdlm {
namespace {

constexpr int BM = kFwdTileRows;  // 64 query rows, 16 per warp
constexpr int BN = kFwdKeyTile;   // 64 keys per step
constexpr int NT = 128;

template <int D>
constexpr int fwd_smem_bytes() {
    return BM * D * 2 + 4 * BN * D * 2;  // Q + 2 stages of K and V
}

template <int D>
__global__ void __launch_bounds__(NT, 2) fwd_mma_kernel(const FwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK0 = sQ + BM * D * 2;
    const uint32_t sV0 = sK0 + 2 * BN * D * 2;
    __shared__ Span s_span[BM];
    __shared__ int s_item;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tq = lane & 3;
    const int H = a.H;
    const int n_items = a.hdr->n_tiles * H;
    const long long q_stride = (long long)H * D;
    const long long k_stride = (long long)a.Hk * D;
    const float sl2 = a.scale_log2;

    for (;;) {
        if (tid == 0) s_item = atomicAdd(&a.hdr->counter, 1);
        __syncthreads();
        const int item = s_item;
        if (item >= n_items) break;
        const Tile t = a.table[item / H];
        const int h = item % H, kvh = h / a.G;
        if (tid < BM) s_span[tid] = row_span(a.lay, t, tid);
        __syncthreads();

        int r1_lo = INT_MAX, r1_hi = 0, r2_lo = INT_MAX, r2_hi = 0, plo_max = 0, phi_min = INT_MAX;
        for (int r = 0; r < t.nrows; ++r) {
            const Span s = s_span[r];
            if (s.p_hi > s.p_lo) {
                r1_lo = imin(r1_lo, s.p_lo);
                r1_hi = imax(r1_hi, s.p_hi);
                plo_max = imax(plo_max, s.p_lo);
                phi_min = imin(phi_min, s.p_hi);
            } else {
                phi_min = 0;
            }
            if (s.d_hi > s.d_lo) {
                r2_lo = imin(r2_lo, s.d_lo);
                r2_hi = imax(r2_hi, s.d_hi);
            }
        }
        const int n1 = r1_hi > r1_lo ? (r1_hi - r1_lo + BN - 1) / BN : 0;
        const int n2 = r2_hi > r2_lo ? (r2_hi - r2_lo + BN - 1) / BN : 0;
        const int nk = n1 + n2;
        const long long q_row0 = (long long)t.doc_start + t.pos0;

        load_tile_async<D, BM, NT>(sQ, a.q, q_row0, q_row0 + t.nrows, q_stride, h);
        cp_async_commit();
        auto key0 = [&](int j) { return j < n1 ? r1_lo + j * BN : r2_lo + (j - n1) * BN; };
        if (nk > 0) {
            load_tile_async<D, BN, NT>(sK0, a.k, key0(0), a.Lk, k_stride, kvh);
            load_tile_async<D, BN, NT>(sV0, a.v, key0(0), a.Lk, k_stride, kvh);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        uint32_t qf[D / 16][4];
#pragma unroll
        for (int kt = 0; kt < D / 16; ++kt)
            ldsm_x4(qf[kt], sQ + swz<D>(warp * 16 + (lane & 15), 2 * kt + (lane >> 4)));

        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        float acc[D / 8][4];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

        for (int j = 0; j < nk; ++j) {
            const int st = j & 1;
            if (j + 1 < nk) {
                const int kn = key0(j + 1);
                load_tile_async<D, BN, NT>(sK0 + (st ^ 1) * BN * D * 2, a.k, kn, a.Lk, k_stride, kvh);
                load_tile_async<D, BN, NT>(sV0 + (st ^ 1) * BN * D * 2, a.v, kn, a.Lk, k_stride, kvh);
                cp_async_commit();
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const uint32_t sK = sK0 + st * BN * D * 2, sV = sV0 + st * BN * D * 2;
            const int k0 = key0(j);
            const bool full = j < n1 && k0 >= plo_max && k0 + BN <= phi_min;

            float s[BN / 8][4];
#pragma unroll
            for (int i = 0; i < BN / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
            for (int kt = 0; kt < D / 16; ++kt) {
#pragma unroll
                for (int p = 0; p < BN / 16; ++p) {
                    uint32_t b[4];
                    ldsm_x4(b, sK + swz<D>(16 * p + (lane >> 4) * 8 + (lane & 7), 2 * kt + ((lane >> 3) & 1)));
                    mma_bf16(s[2 * p], qf[kt], b[0], b[1]);
                    mma_bf16(s[2 * p + 1], qf[kt], b[2], b[3]);
                }
            }
            if (!full) {
                const Span sp0 = s_span[warp * 16 + g], sp1 = s_span[warp * 16 + g + 8];
#pragma unroll
                for (int nt = 0; nt < BN / 8; ++nt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int kr = k0 + nt * 8 + 2 * tq + (e & 1);
                        if (!span_sees(e < 2 ? sp0 : sp1, kr)) s[nt][e] = -INFINITY;
                    }
                }
            }
            // online softmax, base 2
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < BN / 8; ++nt) mx = fmaxf(mx, fmaxf(s[nt][2 * i], s[nt][2 * i + 1]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m[i], mx * sl2);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = fast_exp2(m[i] - m_use);
                float sum = 0.f;
#pragma unroll
                for (int nt = 0; nt < BN / 8; ++nt) {
                    const float p0 = fast_exp2(fmaf(s[nt][2 * i], sl2, -m_use));
                    const float p1 = fast_exp2(fmaf(s[nt][2 * i + 1], sl2, -m_use));
                    s[nt][2 * i] = p0;
                    s[nt][2 * i + 1] = p1;
                    sum += p0 + p1;
                }
                l[i] = l[i] * alpha + sum;
                m[i] = m_new;
#pragma unroll
                for (int dn = 0; dn < D / 8; ++dn) {
                    acc[dn][2 * i] *= alpha;
                    acc[dn][2 * i + 1] *= alpha;
                }
            }
            // O += P V
#pragma unroll
            for (int kc = 0; kc < BN / 16; ++kc) {
                uint32_t pa[4];
                pa[0] = pack_bf16(s[2 * kc][0], s[2 * kc][1]);
                pa[1] = pack_bf16(s[2 * kc][2], s[2 * kc][3]);
                pa[2] = pack_bf16(s[2 * kc + 1][0], s[2 * kc + 1][1]);
                pa[3] = pack_bf16(s[2 * kc + 1][2], s[2 * kc + 1][3]);
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    uint32_t b[4];
                    ldsm_x4_t(b, sV + swz<D>(16 * kc + ((lane >> 3) & 1) * 8 + (lane & 7), 2 * dp + (lane >> 4)));
                    mma_bf16(acc[2 * dp], pa, b[0], b[1]);
                    mma_bf16(acc[2 * dp + 1], pa, b[2], b[3]);
                }
            }
            __syncthreads();
        }

        // epilogue: o = acc / l, lse = ln2 * (m + log2 l)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float li = l[i];
            li += __shfl_xor_sync(0xffffffffu, li, 1);
            li += __shfl_xor_sync(0xffffffffu, li, 2);
            const int r = warp * 16 + g + 8 * i;
            const float inv = li > 0.f ? 1.f / li : 0.f;
            if (r < t.nrows) {
                __nv_bfloat16* orow = a.o + (q_row0 + r) * q_stride + (long long)h * D;
#pragma unroll
                for (int dn = 0; dn < D / 8; ++dn) {
                    const uint32_t v = pack_bf16(acc[dn][2 * i] * inv, acc[dn][2 * i + 1] * inv);
                    *reinterpret_cast<uint32_t*>(orow + dn * 8 + 2 * tq) = v;
                }
                if (tq == 0)
                    a.lse[(long long)h * a.Lq + q_row0 + r] =
                        li > 0.f ? (m[i] + __log2f(li)) * 0.69314718055994531f : -INFINITY;
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, int num_sms, cudaStream_t st, int* launches) {
    cudaError_t e;
    if (a.D == 128) {
        constexpr int smem = fwd_smem_bytes<128>();
        e = cudaFuncSetAttribute(fwd_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        fwd_mma_kernel<128><<<num_sms * 2, NT, smem, st>>>(a);
    } else {
        constexpr int smem = fwd_smem_bytes<64>();
        e = cudaFuncSetAttribute(fwd_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        fwd_mma_kernel<64><<<num_sms * 2, NT, smem, st>>>(a);
    }
    ++*launches;
    return cudaGetLastError();
}

}  // namespace bdlm
