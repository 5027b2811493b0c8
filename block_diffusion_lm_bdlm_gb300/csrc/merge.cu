// merge.cu - log-sum-exp merge of partial attention results.
//
// Partials computed against disjoint key sets (clean-K/V shards and the local
// corrupted keys, as under context-sharded block parallelism) combine into the
// unsharded result: m = max_p lse_p, w_p = exp(lse_p - m), lse = m + ln sum w,
// o = sum w_p o_p / sum w_p. A -inf partial is dropped by selection.
//
// One CTA owns a run of R consecutive rows and all H heads, i.e. one
// contiguous R*H*d slab of every partial. Phase 1: one thread per (head, row)
// reads the P lse values (consecutive rows in consecutive threads, so the
// [H, rows] loads coalesce), writes the merged lse and parks the normalised
// weights in shared memory. Phase 2: the slab is streamed in 16-byte chunks,
// 8 partial loads in flight per thread, weighted in fp32, stored as bf16.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace bdlm {
namespace {

constexpr int MT = 256;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], uint4 x, float w) {
    const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(u[i] << 16);
        const float hi = __uint_as_float(u[i] & 0xffff0000u);
        acc[2 * i] = w > 0.f ? fmaf(w, lo, acc[2 * i]) : acc[2 * i];
        acc[2 * i + 1] = w > 0.f ? fmaf(w, hi, acc[2 * i + 1]) : acc[2 * i + 1];
    }
}

__device__ __forceinline__ void add_f32x4(float* acc, uint4 x, float w) {
    const float f[4] = {__uint_as_float(x.x), __uint_as_float(x.y), __uint_as_float(x.z), __uint_as_float(x.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = w > 0.f ? fmaf(w, f[i], acc[i]) : acc[i];
}

template <int D, bool F32>
__global__ void __launch_bounds__(MT) merge_kernel(const MergeArgs a) {
    extern __shared__ float s_w[];  // [P][MT]
    const int H = a.H;
    const int R = MT / H;            // rows per CTA
    const long long r0 = (long long)blockIdx.x * R;
    const int P = a.P;

    // phase 1: weights
    {
        const int tid = threadIdx.x;
        const int h = tid / R, r = tid % R;
        const long long row = r0 + r;
        if (h < H && row < a.rows) {
            const long long idx = (long long)h * a.rows + row;
            float m = -INFINITY;
            for (int p = 0; p < P; ++p) m = fmaxf(m, __ldg(a.lse_in[p] + idx));
            float sum = 0.f;
            if (m != -INFINITY) {
                for (int p = 0; p < P; ++p) {
                    const float x = __ldg(a.lse_in[p] + idx);
                    const float w = x == -INFINITY ? 0.f : __expf(x - m);
                    s_w[p * MT + tid] = w;
                    sum += w;
                }
                const float inv = 1.f / sum;
                for (int p = 0; p < P; ++p) s_w[p * MT + tid] *= inv;
                a.lse[idx] = m + __logf(sum);
            } else {
                for (int p = 0; p < P; ++p) s_w[p * MT + tid] = 0.f;
                a.lse[idx] = -INFINITY;
            }
        }
    }
    __syncthreads();

    // phase 2: weighted sum of the slab
    constexpr int CH = D / 8;  // 16-byte bf16 output chunks per (row, head)
    const long long slab0 = r0 * H * CH;
    const long long rows_here = (a.rows - r0) < R ? (a.rows - r0) : R;
    const int n_chunks = (int)(rows_here * H * CH);
    for (int c = threadIdx.x; c < n_chunks; c += MT) {
        const int pair = c / CH;               // row-major (row, head) inside the slab
        const int r = pair / H, h = pair % H;
        const int widx = h * R + r;
        const long long gc = slab0 + c;        // global chunk index
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        int p = 0;
        for (; p + 8 <= P; p += 8) {
            uint4 x[8], y[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (F32) {
                    const float* src = static_cast<const float*>(a.part[p + u]) + gc * 8;
                    x[u] = ld_stream(src);
                    y[u] = ld_stream(src + 4);
                } else {
                    x[u] = ld_stream(static_cast<const __nv_bfloat16*>(a.part[p + u]) + gc * 8);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float w = s_w[(p + u) * MT + widx];
                if (F32) {
                    add_f32x4(acc, x[u], w);
                    add_f32x4(acc + 4, y[u], w);
                } else {
                    add_bf16x8(acc, x[u], w);
                }
            }
        }
        for (; p < P; ++p) {
            const float w = s_w[p * MT + widx];
            if (F32) {
                const float* src = static_cast<const float*>(a.part[p]) + gc * 8;
                add_f32x4(acc, ld_stream(src), w);
                add_f32x4(acc + 4, ld_stream(src + 4), w);
            } else {
                add_bf16x8(acc, ld_stream(static_cast<const __nv_bfloat16*>(a.part[p]) + gc * 8), w);
            }
        }
        uint4 out;
        __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[0], acc[1]);
        __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[2], acc[3]);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[4], acc[5]);
        __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[6], acc[7]);
        out.x = *reinterpret_cast<uint32_t*>(&b0);
        out.y = *reinterpret_cast<uint32_t*>(&b1);
        out.z = *reinterpret_cast<uint32_t*>(&b2);
        out.w = *reinterpret_cast<uint32_t*>(&b3);
        __stcs(reinterpret_cast<uint4*>(a.o) + gc, out);
    }
}

template <int D, bool F32>
cudaError_t launch_merge_t(const MergeArgs& a, cudaStream_t st) {
    const int R = MT / a.H;
    const long long grid = (a.rows + R - 1) / R;
    const int smem = a.P * MT * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(merge_kernel<D, F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    merge_kernel<D, F32><<<(unsigned)grid, MT, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, int /*num_sms*/, cudaStream_t st, int* launches) {
    cudaError_t e;
    if (a.D == 128)
        e = a.f32 ? launch_merge_t<128, true>(a, st) : launch_merge_t<128, false>(a, st);
    else
        e = a.f32 ? launch_merge_t<64, true>(a, st) : launch_merge_t<64, false>(a, st);
    if (e == cudaSuccess) ++*launches;
    return e;
}

}  // namespace bdlm
