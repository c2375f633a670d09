// The whole MoE layer for one or two decode tokens in ONE cooperative launch:
// router GEMV -> top-k -> bucketing -> gate/up + SwiGLU -> down + weighted
// combine, Q8_0 or Q4_0 experts ("router -> resident expert -> combine ->
// next layer", amalgafy.com/technical-overview, "Warm target path").
//
// At T = 1 a layer moves ~41 MB and the separate kernels spend much of their
// time in launch ramps, prologues that must first learn the routed experts,
// and tails.  Here one persistent CTA per SM runs every stage; stages that
// need all CTAs' results are separated by a grid barrier (all CTAs are
// co-resident by construction of the cooperative launch):
//   1. every warp computes router logits for a slice of the experts (the
//      1 MiB router streams through all SMs at once)        -> barrier
//   2. every CTA redundantly runs the top-k and the bucketing from the logits
//      (a few KB), so no further barrier is needed to learn the experts
//   3. gate/up items stream through per-warp cp.async rings (as in the
//      separate kernels); the first down items are put in flight before the
//      barrier, since Wd does not depend on h                 -> barrier
//   4. down items, combined into out with fp32 atomics.
// Barrier waits are bounded (MOE_STATUS_TIMEOUT on expiry) and the barrier
// words are cleared by the host with an async memset before every launch.
#include "common.cuh"
#include "pipeline.cuh"
#include "route_warp.cuh"
#include "stream_common.cuh"

namespace moe {

namespace {

using namespace stream;

constexpr int kFuNW = 12;
constexpr int kFuNSTG = 3;
constexpr int kFuThreads = kFuNW * 32;
constexpr int kFuMaxT = 2;
constexpr int kFuMaxP = kFuMaxT * MOE_MAX_TOPK;

struct FusedParams {
    const float* x;
    int T, dm, f, E, k, residual;
    const float* Wr;
    const float* bias;
    const int8_t* gqs;
    const uint16_t* gd;
    const int8_t* uqs;
    const uint16_t* ud;
    const int8_t* dqs;
    const uint16_t* dd;
    float* logits;        // [T][E] scratch
    float* h;             // [P][f] scratch
    unsigned int* sync;   // [2] barrier words, zero at launch
    float* out;           // [T][dm]
    int32_t* idx_out;     // [T][k] or null
    float* wts_out;       // [T][k] or null
    int32_t* offsets_out; // [E+1] or null
    int32_t* status;
};

// All CTAs arrive on one counter (release) and wait until it reaches
// target * gridDim.x (acquire); the counter is cleared by the host before the
// launch and only grows, so barrier `target` needs no generation word.
__device__ void grid_barrier(unsigned int* count, unsigned int target, int32_t* status) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int goal = target * gridDim.x;
        __threadfence();
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(count) : "memory");
        const unsigned long long t0 = global_ns();
        for (unsigned int it = 0;; ++it) {
            unsigned int v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
            if (v >= goal) break;
            if ((it & 255u) == 255u && global_ns() - t0 > kWaitDeadlineNs) {
                flag_status(status, MOE_STATUS_TIMEOUT_BIT);
                break;
            }
        }
    }
    __syncthreads();
}

// Per-format geometry.  Q8_0: 16-value chunks, 4-row down items (16 lanes per
// row); Q4_0: 32-value blocks, 8-row down items (8 lanes per row).
template <int FMT>
struct FuFmt {
    static constexpr int kCF4 = FMT ? 8 : 4;         // float4 of activations per 16-byte weight chunk
    static constexpr int kDnRows = FMT ? kDnRowsPerItemQ4 : kDnRowsPerItem;
    static constexpr int kDnLPR = FMT ? 8 : 16;      // lanes per down row
    static __host__ __device__ int gu_bytes(int dm) { return (FMT ? dm : 2 * dm) + 2 * (dm / 16); }
    static __host__ __device__ int dn_bytes(int f) { return kDnRows * (FMT ? f / 2 : f) + kDnRows * (f / 16); }
};

template <int KG, int KD, int G, int FMT>
__global__ void __launch_bounds__(kFuThreads, 1) decode_fused_kernel(FusedParams p) {
    extern __shared__ __align__(128) unsigned char fsm[];
    __shared__ int s_act[MOE_MAX_EXPERTS], s_beg[MOE_MAX_EXPERTS], s_end[MOE_MAX_EXPERTS];
    __shared__ int s_cb[MOE_MAX_EXPERTS + 1], s_n;
    __shared__ int32_t s_idx[kFuMaxP];
    __shared__ float s_val[kFuMaxP];
    __shared__ int32_t s_ptok[kFuMaxP];
    __shared__ float s_pw[kFuMaxP];
    __shared__ __align__(16) float s_lg[kFuMaxT][MOE_MAX_EXPERTS];

    using F = FuFmt<FMT>;
    constexpr int CF4 = F::kCF4;
    constexpr int kXTok4 = KG * CF4 * 32;        // float4 per staged token (gate/up layout)
    constexpr int kHTok4 = KD * CF4 * F::kDnLPR;  // float4 per staged pair (down layout)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = p.T, dm = p.dm, f = p.f, E = p.E, k = p.k;
    const int P = T * k, d4 = dm / 4, f4 = f / 4;
    const int gu_bytes = F::gu_bytes(dm);
    const int dn_bytes = F::dn_bytes(f);
    const int item_bytes = gu_bytes > dn_bytes ? gu_bytes : dn_bytes;
    unsigned char* ring = fsm + (size_t)warp * kFuNSTG * item_bytes;
    float4* act = reinterpret_cast<float4*>(fsm + (size_t)kFuNW * kFuNSTG * item_bytes);  // x, later h

    // 0. this CTA's first router row into registers (it does not depend on x,
    //    so its round trip overlaps the one of x); activations into shared
    //    memory; combine target out = residual ? x : 0
    constexpr int kQ = 2;  // float4 of a router row per thread: d_model <= 2048 -> d4 <= 512 <= 2 * 384
    float4 wv[kQ];
    if (blockIdx.x < E) {
        const float4* wr = reinterpret_cast<const float4*>(p.Wr) + (size_t)blockIdx.x * d4;
#pragma unroll
        for (int u = 0; u < kQ; ++u) {
            const int q = threadIdx.x + u * kFuThreads;
            wv[u] = q < d4 ? __ldg(wr + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    pdl_wait();
    for (int i = threadIdx.x; i < T * d4; i += kFuThreads) {
        const int t = i / d4, q = i - t * d4;
        act[t * kXTok4 + stage_idx<32, CF4>(q)] = __ldcg(reinterpret_cast<const float4*>(p.x) + (size_t)t * d4 + q);
    }
    for (int i = blockIdx.x * kFuThreads + threadIdx.x; i < T * d4; i += gridDim.x * kFuThreads)
        reinterpret_cast<float4*>(p.out)[i] =
            p.residual ? __ldcg(reinterpret_cast<const float4*>(p.x) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();

    // 1. router logits: one expert row per CTA (all CTAs at once), its threads
    //    split K; every load of the row is in flight at once
    for (int e = blockIdx.x; e < E; e += gridDim.x) {
        if (e != blockIdx.x) {  // further rows (E > grid): loaded here
            const float4* wr = reinterpret_cast<const float4*>(p.Wr) + (size_t)e * d4;
#pragma unroll
            for (int u = 0; u < kQ; ++u) {
                const int q = threadIdx.x + u * kFuThreads;
                wv[u] = q < d4 ? __ldg(wr + q) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float acc[kFuMaxT] = {0.f, 0.f};
#pragma unroll
        for (int u = 0; u < kQ; ++u) {
            const int q = threadIdx.x + u * kFuThreads;
            if (q < d4) {
#pragma unroll
                for (int t = 0; t < kFuMaxT; ++t)
                    if (t < T) {
                        const float4 xv = act[t * kXTok4 + stage_idx<32, CF4>(q)];
                        acc[t] = fmaf(wv[u].x, xv.x,
                                      fmaf(wv[u].y, xv.y, fmaf(wv[u].z, xv.z, fmaf(wv[u].w, xv.w, acc[t]))));
                    }
            }
        }
#pragma unroll
        for (int t = 0; t < kFuMaxT; ++t) {
            const float sw = warp_sum(acc[t]);
            if (lane == 0) s_lg[t][warp] = sw;  // per-warp partials (fixed order below)
        }
        __syncthreads();
        if (threadIdx.x < T) {
            float sum = 0.f;
            for (int w2 = 0; w2 < kFuNW; ++w2) sum += s_lg[threadIdx.x][w2];
            p.logits[(size_t)threadIdx.x * E + e] = sum + (p.bias ? __ldg(p.bias + e) : 0.f);
        }
        __syncthreads();
    }
    grid_barrier(p.sync, 1, p.status);

    // 2. top-k of every token, by every CTA redundantly (a few KB of logits)
    for (int i = threadIdx.x; i < T * E; i += kFuThreads) {
        const int t = i / E, e = i - t * E;
        const float v = __ldcg(p.logits + i);
        s_lg[t][e] = v != v ? -INFINITY : v;
    }
    __syncthreads();
    topk_rank_block(&s_lg[0][0], MOE_MAX_EXPERTS, T, E, k, kFuThreads, s_idx, s_val);
    __syncthreads();
    // 3. weights, bucketing and the active-expert list: warp w takes pair
    //    q = w and its lanes hold the other pairs (P <= 32), so every count
    //    is one ballot; chunks are unbounded here, so active expert a is chunk a
    for (int q = warp; q < P; q += kFuNW) {
        const int e = s_idx[q];
        const int e2 = lane < P ? s_idx[lane] : 0x7fffffff;  // lanes >= P: above every expert
        const uint32_t lt = __ballot_sync(0xffffffffu, e2 < e);
        const uint32_t eq = __ballot_sync(0xffffffffu, e2 == e);
        const uint32_t eq_before = eq & ((1u << q) - 1u);
        const uint32_t same = __match_any_sync(0xffffffffu, e2);
        const bool lead = lane < P && __ffs(same) - 1 == lane;  // first pair of its expert
        const uint32_t leads = __ballot_sync(0xffffffffu, lead);
        const uint32_t leads_below = __ballot_sync(0xffffffffu, lead && e2 < e);
        // weight: softmax over the token's k selected logits
        const int t = q / k;
        const float v0 = s_val[t * k];
        const float den = warp_sum(lane < k ? expf(s_val[t * k + lane] - v0) : 0.0f);
        const float w = expf(s_val[q] - v0) / den;
        if (lane == 0) {
            const int r = __popc(lt) + __popc(eq_before);
            s_ptok[r] = t;
            s_pw[r] = w;
            if (eq_before == 0) {
                const int a = __popc(leads_below);
                s_act[a] = e;
                s_beg[a] = __popc(lt);
                s_end[a] = __popc(lt) + __popc(eq);
                s_cb[a] = a;
            }
            if (q == 0) {
                const int n = __popc(leads);
                s_n = n;
                s_cb[n] = n;
            }
            if (blockIdx.x == 0) {
                if (p.idx_out) p.idx_out[q] = e;
                if (p.wts_out) p.wts_out[q] = w;
            }
        }
    }
    if (blockIdx.x == 0 && p.offsets_out) bucket_offsets(s_idx, P, E, kFuThreads, p.offsets_out);
    __syncthreads();

    // 4. gate/up items (one feature each) -> h
    {
        int lo, hi;
        item_range(s_cb[s_n] * f, &lo, &hi);
        auto issue = [&](int i, int st) {
            const int g = i / f, r = i - g * f;
            const size_t row = (size_t)s_act[locate(g, s_cb, s_n)] * f + r;
            if constexpr (FMT == 1)
                gu_issue_item_q4<KG>(ring + (size_t)st * item_bytes, p.gqs, p.uqs, p.gd, p.ud, row, dm, lane);
            else
                gu_issue_item<KG>(ring + (size_t)st * item_bytes, p.gqs, p.uqs, p.gd, p.ud, row, dm, lane);
        };
        auto compute = [&](int i, int st) {
            const int g = i / f, r = i - g * f;
            const int a = locate(g, s_cb, s_n);
            if constexpr (FMT == 1)
                gu_compute_item_q4<KG, G>(ring + (size_t)st * item_bytes, r, s_beg[a], s_end[a], dm, f, lane, act,
                                          s_ptok, p.h);
            else
                gu_compute_item<KG, G, true>(ring + (size_t)st * item_bytes, r, s_beg[a], s_end[a], dm, f, lane,
                                             act, s_ptok, p.h);
        };
        warp_stream<kFuNSTG>(lo + warp, hi, kFuNW, issue, compute);
    }

    // 5. down items: put the first ones in flight, wait for every CTA's h, stage h
    const int nq = dm / F::kDnRows;
    int lo, hi;
    item_range(s_cb[s_n] * nq, &lo, &hi);
    auto dissue = [&](int i, int st) {
        const int g = i / nq, qd = i - g * nq;
        const size_t row0 = (size_t)s_act[locate(g, s_cb, s_n)] * dm + (size_t)qd * F::kDnRows;
        if constexpr (FMT == 1)
            dn_issue_item_q4(ring + (size_t)st * item_bytes, p.dqs, p.dd, row0, f, lane);
        else
            dn_issue_item(ring + (size_t)st * item_bytes, p.dqs, p.dd, row0, f, lane);
    };
    const int first = lo + warp;
    const int n = first < hi ? (hi - first + kFuNW - 1) / kFuNW : 0;
#pragma unroll
    for (int j = 0; j < kFuNSTG - 1; ++j) {
        if (j < n) dissue(first + j * kFuNW, j);
        else cp_async_commit();
    }
    grid_barrier(p.sync, 2, p.status);
    for (int q = threadIdx.x; q < P * f4; q += kFuThreads) {
        const int pp = q / f4, qq = q - pp * f4;
        act[pp * kHTok4 + stage_idx<F::kDnLPR, CF4>(qq)] =
            __ldcg(reinterpret_cast<const float4*>(p.h) + (size_t)pp * f4 + qq);
    }
    __syncthreads();
    const int hl = lane & (F::kDnLPR - 1), sub = lane / F::kDnLPR;
    for (int j = 0; j < n; ++j) {
        const int jn = j + kFuNSTG - 1;
        if (jn < n) dissue(first + jn * kFuNW, jn % kFuNSTG);
        else cp_async_commit();
        cp_async_wait<kFuNSTG - 1>();
        __syncwarp();
        const int i = first + j * kFuNW;
        const int g = i / nq, qd = i - g * nq;
        const int a = locate(g, s_cb, s_n);
        if constexpr (FMT == 1)
            dn_compute_item_q4<KD, G>(ring + (size_t)(j % kFuNSTG) * item_bytes, qd, s_beg[a], s_end[a], f, dm, hl,
                                      sub, act, s_ptok, s_pw, p.out);
        else
            dn_compute_item<KD, G, true>(ring + (size_t)(j % kFuNSTG) * item_bytes, qd, s_beg[a], s_end[a], f, dm,
                                         k, T, hl, sub, act, s_ptok, s_pw, nullptr, nullptr, nullptr, 1, p.out);
        __syncwarp();
    }
    cp_async_wait<0>();
}

int fused_num_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

template <int KG, int KD, int G, int FMT>
cudaError_t launch_fused(const FusedParams& p, cudaStream_t s) {
    using F = FuFmt<FMT>;
    const int gu = F::gu_bytes(p.dm), dn = F::dn_bytes(p.f);
    const size_t ring = (size_t)kFuNW * kFuNSTG * (gu > dn ? gu : dn);
    const size_t xs = (size_t)p.T * KG * F::kCF4 * 32 * 16, hs = (size_t)p.T * p.k * KD * F::kCF4 * F::kDnLPR * 16;
    const size_t smem = ring + (xs > hs ? xs : hs);
    if (smem > 200 * 1024) return cudaErrorInvalidConfiguration;
    auto kern = decode_fused_kernel<KG, KD, G, FMT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFuThreads, smem);
    if (err != cudaSuccess || per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    err = cudaMemsetAsync(p.sync, 0, 2 * sizeof(unsigned int), s);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(fused_num_sms(), 1, 1);
    cfg.blockDim = dim3(kFuThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

bool decode_fused_supported(const moe_layer_w& w, int T) {
    // the routing phase holds all T*k pairs in one warp's lanes; items are
    // whole 16-byte pieces of weights and scales (K % 256 == 0) and whole
    // down items; at most 4 weight chunks per lane
    if (w.wfmt != MOE_WFMT_Q8_0 && w.wfmt != MOE_WFMT_Q4_0) return false;
    if (w.expert_slot) return false;  // weights in expert order only
    const int rows = w.wfmt == MOE_WFMT_Q4_0 ? kDnRowsPerItemQ4 : kDnRowsPerItem;
    return T >= 1 && T <= kFuMaxT && T * w.k <= 32 && w.d_model % 256 == 0 && w.d_ff % 256 == 0 &&
           w.d_model % rows == 0 && w.d_model <= 2048 && w.d_ff <= 1024;
}

cudaError_t launch_decode_fused(const float* x, int T, const moe_layer_w& w, int residual, float* out,
                                int32_t* idx_out, float* wts_out, int32_t* offsets_out, float* logits, float* h,
                                unsigned int* sync, int32_t* status, cudaStream_t s) {
    FusedParams p = {};
    p.x = x;
    p.T = T;
    p.dm = w.d_model;
    p.f = w.d_ff;
    p.E = w.E;
    p.k = w.k;
    p.residual = residual;
    p.Wr = w.router_w;
    p.bias = w.router_bias;
    p.gqs = w.gate.qs;
    p.gd = w.gate.d;
    p.uqs = w.up.qs;
    p.ud = w.up.d;
    p.dqs = w.down.qs;
    p.dd = w.down.d;
    p.logits = logits;
    p.h = h;
    p.sync = sync;
    p.out = out;
    p.idx_out = idx_out;
    p.wts_out = wts_out;
    p.offsets_out = offsets_out;
    p.status = status;
    if (w.wfmt == MOE_WFMT_Q4_0) {
        // blocks per lane: gate/up d_model/1024, down d_ff/256 (rounded up)
        const int kg = (w.d_model / 32 + 31) / 32, kd = (w.d_ff / 32 + 7) / 8;
#define MOE_FUSED_GO4(KG, KD) \
    return T == 1 ? launch_fused<KG, KD, 1, 1>(p, s) : launch_fused<KG, KD, 2, 1>(p, s)
        if (kg == 2 && kd == 3) MOE_FUSED_GO4(2, 3);
        if (kg == 2 && kd == 4) MOE_FUSED_GO4(2, 4);
        if (kg == 2 && kd == 2) MOE_FUSED_GO4(2, 2);
        if (kg == 1 && kd == 2) MOE_FUSED_GO4(1, 2);
        if (kg == 1 && kd == 1) MOE_FUSED_GO4(1, 1);
#undef MOE_FUSED_GO4
        return cudaErrorInvalidConfiguration;
    }
    // chunks per lane: gate/up d_model/512, down d_ff/256 (rounded up)
    const int kg = (w.d_model / 16 + 31) / 32, kd = (w.d_ff / 16 + 15) / 16;
#define MOE_FUSED_GO(KG, KD) \
    return T == 1 ? launch_fused<KG, KD, 1, 0>(p, s) : launch_fused<KG, KD, 2, 0>(p, s)
    if (kg == 4 && kd == 3) MOE_FUSED_GO(4, 3);
    if (kg == 4 && kd == 4) MOE_FUSED_GO(4, 4);
    if (kg == 4 && kd == 2) MOE_FUSED_GO(4, 2);
    if (kg == 4 && kd == 1) MOE_FUSED_GO(4, 1);
    if (kg == 2 && kd == 2) MOE_FUSED_GO(2, 2);
    if (kg == 2 && kd == 1) MOE_FUSED_GO(2, 1);
    if (kg == 1 && kd == 1) MOE_FUSED_GO(1, 1);
#undef MOE_FUSED_GO
    return cudaErrorInvalidConfiguration;
}

}  // namespace moe
