// bwd_prep.cu - BDLM attention backward: the preprocess and dq-convert
// kernels around the tensor-core main kernel of bwd_tc.cu, and the launch of
// all three (after the tile prologue):
//   1. preprocess: D_i = sum_d dO_i * o_i (fp32) per (row, head), and zero the
//      fp32 dq accumulator in the same pass;
//   2. main: bwd_tc.cu (key-major, dK and dV in TMEM, dq added into the fp32
//      accumulator unscaled);
//   3. convert: dq = bf16(softmax scale * accumulator).
#include "common.cuh"
#include "kernels.h"

namespace bdlm {
namespace {

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
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

// dq = bf16(mul * accumulator), mul = the softmax scale (the main kernel
// accumulates dS K unscaled).
template <int D>
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

template <int D>
cudaError_t launch_bwd_t(const BwdArgs& a, int num_sms, cudaStream_t st) {
    const long long pairs = a.Lq * a.H;
    const long long pre_threads = pairs * (D / 8);
    bwd_pre_kernel<D><<<(unsigned)((pre_threads + 255) / 256), 256, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_bwd_tc_main(a, num_sms, st);  // tensor-core main kernel, 128-key tiles
    if (e != cudaSuccess) return e;
    const long long cv = pairs * D / 8;
    bwd_convert_kernel<D><<<(unsigned)((cv + 255) / 256), 256, 0, st>>>(a, a.scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, int num_sms, cudaStream_t st, int* launches) {
    cudaError_t e = a.D == 128 ? launch_bwd_t<128>(a, num_sms, st) : launch_bwd_t<64>(a, num_sms, st);
    if (e == cudaSuccess) *launches += 3;
    return e;
}

}  // namespace bdlm
