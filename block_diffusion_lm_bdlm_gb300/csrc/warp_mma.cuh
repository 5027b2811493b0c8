// warp_mma.cuh - warp-level tensor-core helpers (mma.sync m16n8k16 bf16,
// ldmatrix, cp.async) and the XOR-swizzled shared-memory tile layout they use.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace bdlm {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; copies zeros when !pred.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
    const int sz = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// c += a * b, a 16x16 (row), b 16x8 (col), bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of 16-byte chunk c of row r in a [rows][D] bf16 tile whose
// chunks are XOR-swizzled by (r mod 8), so that the 8 rows one ldmatrix
// reads fall in 8 different bank groups.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

// Asynchronously load rows [row0, row0 + ROWS) of head `head` of a [*, heads, D]
// bf16 tensor into a swizzled tile; rows outside [0, row_end) read as zeros.
template <int D, int ROWS, int NTHREADS>
__device__ __forceinline__ void load_tile_async(uint32_t s_base, const __nv_bfloat16* g, long long row0,
                                                long long row_end, long long row_stride, int head) {
    constexpr int CH = D / 8;
    for (int i = threadIdx.x; i < ROWS * CH; i += NTHREADS) {
        const int r = i / CH, c = i % CH;
        const long long gr = row0 + r;
        const bool ok = gr >= 0 && gr < row_end;
        const __nv_bfloat16* src = ok ? g + gr * row_stride + (long long)head * D + c * 8 : g;
        cp_async16(s_base + swz<D>(r, c), src, ok);
    }
}

}  // namespace bdlm
