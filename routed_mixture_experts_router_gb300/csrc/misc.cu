// Load-time Q8_0 repack and the fixed-order weighted combine.
#include "common.cuh"

namespace moe {

namespace {

// One thread per 34-byte block: fp16 scale (little endian) then 32 int8
// values (amalgafy.com/technical-overview, "Validated GPU foundation":
// native Q8_0 weights).  The scale is copied unchanged; each value q is
// stored as the byte q + 128 (its sign bit flipped: offset binary), the form
// every kernel's exact dequantisation takes directly.
__global__ void pack_q8_kernel(const uint8_t* __restrict__ blocks, long long nblocks, int8_t* __restrict__ qs,
                               uint16_t* __restrict__ d) {
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const uint8_t* src = blocks + b * 34;
    d[b] = (uint16_t)(src[0] | (src[1] << 8));
    uint32_t wv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        wv[i] = ((uint32_t)src[2 + 4 * i] | ((uint32_t)src[3 + 4 * i] << 8) | ((uint32_t)src[4 + 4 * i] << 16) |
                 ((uint32_t)src[5 + 4 * i] << 24)) ^
                0x80808080u;  // q -> q + 128 in every byte
    uint4* dst = reinterpret_cast<uint4*>(qs + b * 32);
    dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
}

// One 18-byte Q4_0 block per thread: the scale to d, the 16 nibble bytes
// unchanged to qs (the device layout keeps the block's own nibble order).
__global__ void pack_q4_kernel(const uint8_t* __restrict__ blocks, long long nblocks, uint8_t* __restrict__ qs,
                               uint16_t* __restrict__ d) {
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const uint8_t* src = blocks + b * 18;
    d[b] = (uint16_t)(src[0] | (src[1] << 8));
    uint32_t wv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        wv[i] = (uint32_t)src[2 + 4 * i] | ((uint32_t)src[3 + 4 * i] << 8) | ((uint32_t)src[4 + 4 * i] << 16) |
                ((uint32_t)src[5 + 4 * i] << 24);
    reinterpret_cast<uint4*>(qs)[b] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
}

// out[t][o] = (residual ? residual[t][o] : 0) + sum_{s<k} wts[t][s] * ypairs[pos[t][s]][o], s ascending.
// ("weighted combine", amalgafy.com/technical-overview, "Execution architecture")
__global__ void combine_kernel(const float* __restrict__ ypairs, const float* __restrict__ wts,
                               const int32_t* __restrict__ pos, int T, int k, int dm4, int P,
                               const float* __restrict__ residual, float* __restrict__ out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)T * dm4) return;
    const int t = (int)(i / dm4), q = (int)(i - (long long)t * dm4);
    float4 acc = residual ? __ldg(reinterpret_cast<const float4*>(residual) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < k; ++s) {
        const int p = __ldg(pos + (size_t)t * k + s);
        if (p < 0 || p >= P) continue;
        const float w = __ldg(wts + (size_t)t * k + s);
        const float4 y = __ldg(reinterpret_cast<const float4*>(ypairs) + (size_t)p * dm4 + q);
        acc.x = fmaf(w, y.x, acc.x);
        acc.y = fmaf(w, y.y, acc.y);
        acc.z = fmaf(w, y.z, acc.z);
        acc.w = fmaf(w, y.w, acc.w);
    }
    reinterpret_cast<float4*>(out)[i] = acc;
}

}  // namespace

cudaError_t launch_pack_q8(const uint8_t* blocks, long long rows, int K, int8_t* qs, uint16_t* d, cudaStream_t s) {
    const long long nb = rows * (K / 32);
    if (nb == 0) return cudaSuccess;
    const int threads = 256;
    const long long grid = (nb + threads - 1) / threads;
    pack_q8_kernel<<<(unsigned)grid, threads, 0, s>>>(blocks, nb, qs, d);
    return cudaGetLastError();
}

cudaError_t launch_pack_q4(const uint8_t* blocks, long long rows, int K, uint8_t* qs, uint16_t* d, cudaStream_t s) {
    const long long nb = rows * (K / 32);
    if (nb == 0) return cudaSuccess;
    const int threads = 256;
    const long long grid = (nb + threads - 1) / threads;
    pack_q4_kernel<<<(unsigned)grid, threads, 0, s>>>(blocks, nb, qs, d);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float* ypairs, const float* wts, const int32_t* pos, int T, int k, int dm,
                           const float* residual, float* out, cudaStream_t s) {
    const long long n = (long long)T * (dm / 4);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    combine_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(ypairs, wts, pos, T, k, dm / 4, T * k,
                                                                               residual, out);
    return cudaGetLastError();
}

}  // namespace moe
