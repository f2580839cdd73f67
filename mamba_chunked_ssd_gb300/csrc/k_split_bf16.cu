// k_split_bf16.cu — fp32 rows to pairs of bf16 rows (hi, lo) for the fp32
// forward pass on the tensor cores.
//
// An fp32 value v is carried as hi = bf16(v) and lo = bf16(v - hi); the
// tensor-core kernels form each fp32 product u v as u_hi v_hi + u_hi v_lo +
// u_lo v_hi, which leaves out u_lo v_lo and the rounding of the lo parts,
// both below 2^-16 |u v|.  Rows of `width` values become two rows, hi then
// lo: x [b, L, nh, H] -> [b, L, nh, 2, H] (a head 2h + 0/1 of 2 nh heads),
// B and C [b, L, G, S] -> [b, L, G, 2, S], chunk states [.., S, H] ->
// [.., 2, S, H].
#include "common.cuh"

namespace m2 {
namespace {

__global__ void __launch_bounds__(256) k_split_rows(const float4* __restrict__ src, uint2* __restrict__ dst,
                                                    int64_t rows, int width4) {
    const int64_t n = rows * width4;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = e / width4, c = e - r * width4;
        const float4 v = src[e];
        const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y), h23 = __floats2bfloat162_rn(v.z, v.w);
        const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
        const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - f01.x, v.y - f01.y);
        const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - f23.x, v.w - f23.y);
        uint2 hi, lo;
        hi.x = *reinterpret_cast<const uint32_t*>(&h01);
        hi.y = *reinterpret_cast<const uint32_t*>(&h23);
        lo.x = *reinterpret_cast<const uint32_t*>(&l01);
        lo.y = *reinterpret_cast<const uint32_t*>(&l23);
        dst[(2 * r) * width4 + c] = hi;
        dst[(2 * r + 1) * width4 + c] = lo;
    }
}

}  // namespace

cudaError_t launch_split_bf16(const float* src, void* dst, int64_t rows, int width, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    const int width4 = width / 4;
    const int64_t n = rows * width4;
    const int64_t blocks = (n + 255) / 256;
    const unsigned grid = (unsigned)(blocks < 152 * 16 ? blocks : 152 * 16);
    k_split_rows<<<grid, 256, 0, st>>>(reinterpret_cast<const float4*>(src), reinterpret_cast<uint2*>(dst), rows,
                                       width4);
    return cudaGetLastError();
}

}  // namespace m2
