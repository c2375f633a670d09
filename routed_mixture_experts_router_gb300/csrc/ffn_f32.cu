// Expert SwiGLU FFNs with fp32 activations (the decode path): Q8_0
// dequantisation fused into CUDA-core contractions, combine fused into the
// down projection.
//
//   gate/up  h[p][r] = silu(Wg_e[r] . x[t]) * (Wu_e[r] . x[t])   for pair p = (t, slot) in bucket e
//   down     y[p][o] = Wd_e[o] . h[p]
//   combine  out[t][o] += w[t][slot] * y[p][o]          (fp32 atomics, fuse_combine = 1)
//            ypairs[p][o] = y[p][o]                      (fuse_combine = 0)
// Q8_0 (amalgafy.com/technical-overview, "Validated GPU foundation": native
// Q8_0 weights); the down projection K=768 -> 2048 rows (expxa.com
// reuse-ordering-qualification, "What changed from the first experiment").
//
// Memory-bound design.  Grid = (row tiles) x (active experts): a CTA owns a
// tile of weight rows of ONE expert and applies it to every token of that
// expert's bucket, so each weight byte is read from HBM once per layer.  A
// group of LPR lanes owns one weight row; its lanes split K in 16-byte chunks
// (16 int8 = half a Q8_0 block), so every load is a coalesced 128-bit
// streaming load.  The whole row is loaded into registers before the bucket's
// activations are staged in shared memory, so weight traffic starts at once.
// Per chunk, the 16 products q*x are summed exactly as integers-times-floats
// and scaled once by the block's fp16 d (w = q*d, then sum w*x is regrouped
// as d * sum q*x over the half block; fp32 throughout).
#include "common.cuh"

namespace moe {

namespace {

constexpr int kFfnThreads = 256;
constexpr int kFfnWarps = kFfnThreads / kWarp;

// Shared-memory layout of one staged activation vector for a group of LPR
// lanes that split K in 16-byte (16-value) chunks c = hl + LPR*i: float4 m of
// chunk c sits at (i*4 + m)*LPR + hl, so the LPR lanes of one load
// instruction read consecutive float4s (no bank conflicts).
template <int LPR>
__device__ __forceinline__ int stage_index(int q /* float4 index in the row */) {
    const int c = q >> 2, m = q & 3;
    const int i = c / LPR, hl = c % LPR;
    return (i * 4 + m) * LPR + hl;
}

// Index of the a-th expert with a non-empty bucket (-1 if none); one warp.
// Buckets are clamped into [0, P]: offsets that are not a valid bucketing
// give wrong sums, never an out-of-range pair.
__device__ __forceinline__ int find_active_expert(const int32_t* offsets, int E, int P, int a, int* beg, int* end) {
    const int lane = threadIdx.x & 31;
    int seen = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int lo = min(max(e < E ? __ldg(offsets + e) : 0, 0), P);
        const int hi = min(max(e < E ? __ldg(offsets + e + 1) : 0, lo), P);
        const uint32_t act = __ballot_sync(0xffffffffu, hi > lo);
        const int n = __popc(act);
        if (a < seen + n) {
            // the (a - seen)-th set bit of act
            int want = a - seen;
            uint32_t m = act;
            for (int i = 0; i < want; ++i) m &= m - 1;
            const int src = __ffs(m) - 1;
            *beg = __shfl_sync(0xffffffffu, lo, src);
            *end = __shfl_sync(0xffffffffu, hi, src);
            return e0 + src;
        }
        seen += n;
    }
    return -1;
}

// ---------------------------------------------------------------- gate/up --
// One warp per output feature r: lanes split K = d_model (LPR = 32), KCH
// chunks per lane.  TC tokens of the bucket per pass.
template <int KCH, int TC>
__global__ void __launch_bounds__(kFfnThreads, 2) gateup_f32_kernel(
    const float* __restrict__ x, int T, int dm, int f, int E, const int8_t* __restrict__ gqs,
    const uint16_t* __restrict__ gd, const int8_t* __restrict__ uqs, const uint16_t* __restrict__ ud,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_tok, float* __restrict__ h,
    float* __restrict__ out_init, int init_residual, int P) {
    extern __shared__ float4 gu_smem[];  // [TC][KCH*4*32] float4
    __shared__ int s_e, s_beg, s_end;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kTok4 = KCH * 4 * 32;  // float4 per staged token
    const int nch = dm / 16;

    // Initialise the combine target (grid-stride; the down kernel runs after this one).
    if (out_init) {
        const size_t n4 = (size_t)T * dm / 4;
        const size_t nblk = (size_t)gridDim.x * gridDim.y;
        const size_t b = (size_t)blockIdx.y * gridDim.x + blockIdx.x;
        float4* o4 = reinterpret_cast<float4*>(out_init);
        const float4* x4 = reinterpret_cast<const float4*>(x);
        for (size_t i = b * kFfnThreads + threadIdx.x; i < n4; i += nblk * kFfnThreads)
            o4[i] = init_residual ? __ldg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (warp == 0) {
        int beg = 0, end = 0;
        const int e = find_active_expert(offsets, E, P, blockIdx.y, &beg, &end);
        if (lane == 0) {
            s_e = e;
            s_beg = beg;
            s_end = end;
        }
    }
    __syncthreads();
    const int e = s_e;
    if (e < 0) return;
    const int beg = s_beg, end = s_end;
    const int r = blockIdx.x * kFfnWarps + warp;
    const bool row_ok = r < f;

    // the weight row (gate and up) into registers
    uint4 gq[KCH], uq[KCH];
    float gs[KCH], us[KCH];
    const size_t row = (size_t)e * f + (row_ok ? r : 0);
#pragma unroll
    for (int i = 0; i < KCH; ++i) {
        const int c = lane + 32 * i;
        if (row_ok && c < nch) {
            gq[i] = ldg_stream16(gqs + row * dm + (size_t)c * 16);
            uq[i] = ldg_stream16(uqs + row * dm + (size_t)c * 16);
            gs[i] = ldg_half(gd + row * (dm / 32) + (c >> 1));
            us[i] = ldg_half(ud + row * (dm / 32) + (c >> 1));
        } else {
            gq[i] = make_uint4(0, 0, 0, 0);
            uq[i] = make_uint4(0, 0, 0, 0);
            gs[i] = 0.f;
            us[i] = 0.f;
        }
    }

    for (int p0 = beg; p0 < end; p0 += TC) {
        const int n = min(TC, end - p0);
        __syncthreads();  // previous pass finished reading the staged tokens
        const int d4 = dm / 4;
        for (int i = threadIdx.x; i < n * d4; i += kFfnThreads) {
            const int j = i / d4, q = i - j * d4;
            const int t = __ldg(pair_tok + p0 + j);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t >= 0 && t < T) v = __ldg(reinterpret_cast<const float4*>(x) + (size_t)t * d4 + q);
            gu_smem[j * kTok4 + stage_index<32>(q)] = v;
        }
        __syncthreads();
        float ga[TC], ua[TC];
#pragma unroll
        for (int t = 0; t < TC; ++t) {
            ga[t] = 0.f;
            ua[t] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < KCH; ++i) {
            const int c = lane + 32 * i;
            if (c < nch) {
                float gp[TC], up[TC];
#pragma unroll
                for (int t = 0; t < TC; ++t) {
                    gp[t] = 0.f;
                    up[t] = 0.f;
                }
                const uint32_t gw[4] = {gq[i].x, gq[i].y, gq[i].z, gq[i].w};
                const uint32_t uw[4] = {uq[i].x, uq[i].y, uq[i].z, uq[i].w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 gf = i8x4_to_f32x4(gw[m]);
                    const float4 uf = i8x4_to_f32x4(uw[m]);
#pragma unroll
                    for (int t = 0; t < TC; ++t) {
                        if (t < n) {
                            const float4 xv = gu_smem[t * kTok4 + (i * 4 + m) * 32 + lane];
                            gp[t] = dot4(gf, xv, gp[t]);
                            up[t] = dot4(uf, xv, up[t]);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < TC; ++t) {
                    ga[t] = fmaf(gs[i], gp[t], ga[t]);
                    ua[t] = fmaf(us[i], up[t], ua[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TC; ++t) {
            ga[t] = warp_sum(ga[t]);
            ua[t] = warp_sum(ua[t]);
        }
        if (row_ok) {
#pragma unroll
            for (int t = 0; t < TC; ++t)
                if (lane == t && t < n) h[(size_t)(p0 + t) * f + r] = silu_f(ga[t]) * ua[t];
        }
    }
}

// ------------------------------------------------------------------- down --
// LPR lanes per output row o (K = d_ff), 32/LPR rows per warp.
template <int LPR, int KCH, int TC>
__global__ void __launch_bounds__(kFfnThreads, 2) down_f32_kernel(
    const float* __restrict__ h, int T, int f, int dm, int E, int k, const int8_t* __restrict__ dqs,
    const uint16_t* __restrict__ dd, const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_tok,
    const int32_t* __restrict__ pair_slot, const float* __restrict__ wts, int fuse, float* __restrict__ out) {
    extern __shared__ float4 dn_smem[];  // [TC][KCH*4*LPR] float4
    __shared__ int s_e, s_beg, s_end;
    constexpr int kRowsPerWarp = 32 / LPR;
    constexpr int kTok4 = KCH * 4 * LPR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hl = lane % LPR, sub = lane / LPR;
    const int nch = f / 16;
    if (warp == 0) {
        int beg = 0, end = 0;
        const int e = find_active_expert(offsets, E, T * k, blockIdx.y, &beg, &end);
        if (lane == 0) {
            s_e = e;
            s_beg = beg;
            s_end = end;
        }
    }
    __syncthreads();
    const int e = s_e;
    if (e < 0) return;
    const int beg = s_beg, end = s_end;
    const int o = (blockIdx.x * kFfnWarps + warp) * kRowsPerWarp + sub;
    const bool row_ok = o < dm;
    const size_t row = (size_t)e * dm + (row_ok ? o : 0);

    uint4 wq[KCH];
    float ws[KCH];
#pragma unroll
    for (int i = 0; i < KCH; ++i) {
        const int c = hl + LPR * i;
        if (row_ok && c < nch) {
            wq[i] = ldg_stream16(dqs + row * f + (size_t)c * 16);
            ws[i] = ldg_half(dd + row * (f / 32) + (c >> 1));
        } else {
            wq[i] = make_uint4(0, 0, 0, 0);
            ws[i] = 0.f;
        }
    }

    for (int p0 = beg; p0 < end; p0 += TC) {
        const int n = min(TC, end - p0);
        __syncthreads();
        const int f4 = f / 4;
        for (int i = threadIdx.x; i < n * f4; i += kFfnThreads) {
            const int j = i / f4, q = i - j * f4;
            dn_smem[j * kTok4 + stage_index<LPR>(q)] =
                __ldg(reinterpret_cast<const float4*>(h) + (size_t)(p0 + j) * f4 + q);
        }
        __syncthreads();
        float acc[TC];
#pragma unroll
        for (int t = 0; t < TC; ++t) acc[t] = 0.f;
#pragma unroll
        for (int i = 0; i < KCH; ++i) {
            const int c = hl + LPR * i;
            if (c < nch) {
                float part[TC];
#pragma unroll
                for (int t = 0; t < TC; ++t) part[t] = 0.f;
                const uint32_t ww[4] = {wq[i].x, wq[i].y, wq[i].z, wq[i].w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 wf = i8x4_to_f32x4(ww[m]);
#pragma unroll
                    for (int t = 0; t < TC; ++t)
                        if (t < n) part[t] = dot4(wf, dn_smem[t * kTok4 + (i * 4 + m) * LPR + hl], part[t]);
                }
#pragma unroll
                for (int t = 0; t < TC; ++t) acc[t] = fmaf(ws[i], part[t], acc[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < TC; ++t) acc[t] = group_sum<LPR>(acc[t]);
        if (row_ok) {
#pragma unroll
            for (int t = 0; t < TC; ++t) {
                if (hl == t && t < n) {
                    const int p = p0 + t;
                    if (fuse) {
                        const int tok = __ldg(pair_tok + p), s = __ldg(pair_slot + p);
                        if (tok >= 0 && tok < T && s >= 0 && s < k)
                            atomicAdd(out + (size_t)tok * dm + o, __ldg(wts + (size_t)tok * k + s) * acc[t]);
                    } else {
                        out[(size_t)p * dm + o] = acc[t];
                    }
                }
            }
        }
    }
}

template <int KCH, int TC>
cudaError_t launch_gateup(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                          const int32_t* pair_tok, float* h, float* out_init, int residual, cudaStream_t s) {
    const int P = T * w.k;
    const size_t smem = (size_t)TC * KCH * 4 * 32 * sizeof(float4);
    auto kern = gateup_f32_kernel<KCH, TC>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid((w.d_ff + kFfnWarps - 1) / kFfnWarps, P < w.E ? P : w.E);
    kern<<<grid, kFfnThreads, smem, s>>>(x, T, w.d_model, w.d_ff, w.E, w.gate.qs, w.gate.d, w.up.qs, w.up.d, offsets,
                                         pair_tok, h, out_init, residual, P);
    return cudaGetLastError();
}

template <int LPR, int KCH, int TC>
cudaError_t launch_down(const float* h, int T, const moe_layer_w& w, const int32_t* offsets, const int32_t* pair_tok,
                        const int32_t* pair_slot, const float* wts, int fuse, float* out, cudaStream_t s) {
    const int P = T * w.k;
    const size_t smem = (size_t)TC * KCH * 4 * LPR * sizeof(float4);
    auto kern = down_f32_kernel<LPR, KCH, TC>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    constexpr int kRowsPerCta = kFfnWarps * (32 / LPR);
    dim3 grid((w.d_model + kRowsPerCta - 1) / kRowsPerCta, P < w.E ? P : w.E);
    kern<<<grid, kFfnThreads, smem, s>>>(h, T, w.d_ff, w.d_model, w.E, w.k, w.down.qs, w.down.d, offsets, pair_tok,
                                         pair_slot, wts, fuse, out);
    return cudaGetLastError();
}

template <int TC>
cudaError_t dispatch_gateup(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                            const int32_t* pair_tok, float* h, float* out_init, int residual, cudaStream_t s) {
    const int kch = (w.d_model / 16 + 31) / 32;
    switch (kch) {
        case 1: return launch_gateup<1, TC>(x, T, w, offsets, pair_tok, h, out_init, residual, s);
        case 2: return launch_gateup<2, TC>(x, T, w, offsets, pair_tok, h, out_init, residual, s);
        case 3: return launch_gateup<3, TC>(x, T, w, offsets, pair_tok, h, out_init, residual, s);
        case 4: return launch_gateup<4, TC>(x, T, w, offsets, pair_tok, h, out_init, residual, s);
        default:
            if (kch <= 8) return launch_gateup<8, TC>(x, T, w, offsets, pair_tok, h, out_init, residual, s);
            if (kch <= 16) return launch_gateup<16, TC>(x, T, w, offsets, pair_tok, h, out_init, residual, s);
            return cudaErrorInvalidValue;
    }
}

template <int TC>
cudaError_t dispatch_down(const float* h, int T, const moe_layer_w& w, const int32_t* offsets,
                          const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse, float* out,
                          cudaStream_t s) {
    const int nch = w.d_ff / 16;
    if (nch <= 16) return launch_down<16, 1, TC>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, s);
    if (nch <= 32) return launch_down<16, 2, TC>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, s);
    if (nch <= 48) return launch_down<16, 3, TC>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, s);
    if (nch <= 128) return launch_down<32, 4, TC>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, s);
    if (nch <= 256) return launch_down<32, 8, TC>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, s);
    if (nch <= 512) return launch_down<32, 16, TC>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, s);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_ffn_f32(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                           const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse_combine,
                           float* out_or_ypairs, int residual, float* h, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    float* out_init = fuse_combine ? out_or_ypairs : nullptr;
    cudaError_t err;
    if (T == 1) {
        err = dispatch_gateup<1>(x, T, w, offsets, pair_tok, h, out_init, residual, s);
        if (err != cudaSuccess) return err;
        return dispatch_down<1>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs, s);
    }
    err = dispatch_gateup<4>(x, T, w, offsets, pair_tok, h, out_init, residual, s);
    if (err != cudaSuccess) return err;
    return dispatch_down<4>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs, s);
}

}  // namespace moe
