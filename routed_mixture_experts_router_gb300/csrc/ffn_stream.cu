// Expert SwiGLU FFNs with fp32 activations, streaming design (decode path).
//
//   gate/up  h[p][r] = silu(Wg_e[r] . x[t]) * (Wu_e[r] . x[t])   pair p = (t, slot) in bucket e
//   down     y[p][o] = Wd_e[o] . h[p];  out[t][o] += w[t][slot] * y[p][o]  (combine fused)
// Q8_0 weights w = q * d (amalgafy.com/technical-overview, "Validated GPU
// foundation"); down projection K=768 -> 2048 rows (expxa.com
// reuse-ordering-qualification, "What changed from the first experiment");
// weighted combine ("Execution architecture", amalgafy.com/technical-overview).
//
// HBM-bound design for GB300.  A persistent grid of one CTA per SM walks a
// contiguous range of work items: one output feature (its gate row and up
// row) for gate/up, four rows for down, always of one expert.  Every warp owns
// a private ring of NSTG shared-memory stages and streams its items into it
// with 16-byte asynchronous copies (cp.async.cg: L2 -> shared, no registers),
// NSTG - 1 items ahead of the one it computes, so 100+ KB per SM stay in
// flight -- the bandwidth-latency product GB300's HBM needs.  (A ring fed by
// 1-D bulk copies was measured slower: each bulk copy has a fixed cost that
// small Q8_0 rows cannot amortise.)  The activations of the tokens routed to
// the expert sit in shared memory.  Each weight byte is read from HBM once per
// layer.
//
// Arithmetic: int8 -> fp32 exactly (byte placed in the mantissa of 2^23, then
// 2^23 + 128 subtracted), products and sums in fp32 with Blackwell's paired
// fp32 FMA (fma.rn.f32x2), the fp16 block scale applied once per 16-value half
// block.  The down kernel is a programmatic dependent of gate/up: it starts
// streaming Wd before gate/up finishes and waits only before reading h.
#include "common.cuh"
#include "pipeline.cuh"
#include "stream_common.cuh"

namespace moe {

namespace {

using namespace stream;

// ============================================================== gate / up ==
// One warp per output feature r (its gate row and up row); lanes split
// K = d_model in 16-byte chunks c = lane + 32*m, m < KCH.  G: tokens per
// register block; ALLTOK: every token's x staged once (T small), else per
// bucket chunk of at most tca pairs.
template <int KCH, int G, bool ALLTOK, int NW, int NSTG>
__global__ void __launch_bounds__(NW * 32, 1) gateup_cp_kernel(
    const float* __restrict__ x, int T, int dm, int f, int E, const int8_t* __restrict__ gqs,
    const uint16_t* __restrict__ gd, const int8_t* __restrict__ uqs, const uint16_t* __restrict__ ud,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_tok, float* __restrict__ h,
    float* __restrict__ out_init, int init_residual, int tca, int P, const int32_t* __restrict__ eslot,
    int nslots) {
    extern __shared__ __align__(128) unsigned char gu_smem[];
    __shared__ int s_act[MOE_MAX_EXPERTS], s_beg[MOE_MAX_EXPERTS], s_end[MOE_MAX_EXPERTS];
    __shared__ int s_cb[MOE_MAX_EXPERTS + 1], s_n;
    __shared__ int s_tok[ALLTOK ? kMaxStagedPairs : 1];
    __shared__ int s_segtok[ALLTOK ? 1 : kMaxStagedPairs];
    constexpr int kThreads = NW * 32;
    constexpr int kTok4 = KCH * 4 * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d4 = dm / 4;
    const int item_bytes = 2 * dm + 2 * (dm / 16);  // gate qs, up qs, gate d, up d
    unsigned char* ring = gu_smem + (size_t)warp * NSTG * item_bytes;
    float4* xs = reinterpret_cast<float4*>(gu_smem + (size_t)NW * NSTG * item_bytes);

    pdl_wait();  // routing / bucketing of this layer complete and visible
    if (warp == 0)
        build_active(offsets, E, ALLTOK ? (1 << 30) : tca, P, s_act, s_beg, s_end, s_cb, &s_n, eslot, nslots);
    if (ALLTOK) {
        for (int p = threadIdx.x; p < P; p += kThreads) {
            const int t = __ldcg(pair_tok + p);
            s_tok[p] = (t >= 0 && t < T) ? t : 0;
        }
        for (int i = threadIdx.x; i < T * d4; i += kThreads) {
            const int t = i / d4, q = i - t * d4;
            xs[t * kTok4 + stage_idx<32>(q)] = __ldcg(reinterpret_cast<const float4*>(x) + (size_t)t * d4 + q);
        }
    }
    if (out_init) {  // combine target: (residual ? x : 0), consumed by the down kernel
        const size_t n4 = (size_t)T * d4;
        float4* o4 = reinterpret_cast<float4*>(out_init);
        const float4* x4 = reinterpret_cast<const float4*>(x);
        for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < n4; i += (size_t)gridDim.x * kThreads)
            o4[i] = init_residual ? __ldcg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    pdl_launch_dependents();
    int lo, hi;
    item_range(s_cb[s_n] * f, &lo, &hi);

    // item i = (global chunk i / f, feature i % f)
    auto issue = [&](int i, int st) {
        const int g = i / f, r = i - g * f;
        gu_issue_item<KCH>(ring + (size_t)st * item_bytes, gqs, uqs, gd, ud,
                           (size_t)s_act[locate(g, s_cb, s_n)] * f + r, dm, lane);
    };
    auto compute = [&](int i, int st) {
        const int g = i / f, r = i - g * f;
        const int a = locate(g, s_cb, s_n);
        const int c0 = g - s_cb[a];
        const int pb = ALLTOK ? s_beg[a] : s_beg[a] + c0 * tca;
        const int pe = ALLTOK ? s_end[a] : min(s_end[a], pb + tca);
        if constexpr (G == kMultiG)
            gu_compute_multi<KCH, ALLTOK>(ring + (size_t)st * item_bytes, r, pb, pe, dm, f, lane, xs, s_tok, h);
        else
            gu_compute_item<KCH, G, ALLTOK>(ring + (size_t)st * item_bytes, r, pb, pe, dm, f, lane, xs, s_tok, h);
    };

    if (ALLTOK) {
        warp_stream<NSTG>(lo + warp, hi, NW, issue, compute);
    } else {
        for (int seg = lo; seg < hi;) {
            const int g = seg / f;
            const int seg_end = min(hi, (g + 1) * f);
            const int a = locate(g, s_cb, s_n);
            const int pb = s_beg[a] + (g - s_cb[a]) * tca;
            const int pe = min(s_end[a], pb + tca);
            __syncthreads();  // the previous segment's activations are no longer read
            for (int j = threadIdx.x; j < pe - pb; j += kThreads) s_segtok[j] = __ldcg(pair_tok + pb + j);
            __syncthreads();
#pragma unroll 4
            for (int q = threadIdx.x; q < (pe - pb) * d4; q += kThreads) {
                const int jj = q / d4, qq = q - jj * d4;
                const int t = s_segtok[jj];
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t >= 0 && t < T) v = __ldcg(reinterpret_cast<const float4*>(x) + (size_t)t * d4 + qq);
                xs[jj * kTok4 + stage_idx<32>(qq)] = v;
            }
            __syncthreads();
            warp_stream<NSTG>(seg + warp, seg_end, NW, issue, compute);
            seg = seg_end;
        }
    }
    cp_async_wait<0>();
}

// =================================================================== down ==
// An item is 4 consecutive rows (2 per half-warp, LPR = 16 lanes per row);
// lanes split K = d_ff in 16-byte chunks c = hl + 16*m, m < KCH.
// ALLP: every pair's h staged once, else per bucket chunk of at most tcp.
template <int KCH, int G, bool ALLP, int NW, int NSTG>
__global__ void __launch_bounds__(NW * 32, 1) down_cp_kernel(
    const float* __restrict__ h, int T, int f, int dm, int E, int k, const int8_t* __restrict__ dqs,
    const uint16_t* __restrict__ dd, const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_tok,
    const int32_t* __restrict__ pair_slot, const float* __restrict__ wts, int fuse, float* __restrict__ out,
    int tcp, const int32_t* __restrict__ eslot, int nslots) {
    extern __shared__ __align__(128) unsigned char dn_smem[];
    __shared__ int s_act[MOE_MAX_EXPERTS], s_beg[MOE_MAX_EXPERTS], s_end[MOE_MAX_EXPERTS];
    __shared__ int s_cb[MOE_MAX_EXPERTS + 1], s_n;
    __shared__ int s_ptok[ALLP ? kMaxStagedPairs : 1];
    __shared__ float s_pw[ALLP ? kMaxStagedPairs : 1];
    __shared__ int s_segtok[ALLP ? 1 : kMaxStagedPairs];
    __shared__ float s_segw[ALLP ? 1 : kMaxStagedPairs];
    constexpr int kThreads = NW * 32;
    constexpr int LPR = 16;
    constexpr int kTok4 = KCH * 4 * LPR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hl = lane & 15, sub = lane >> 4;
    const int f4 = f / 4;
    const int P = T * k;
    const int nq = dm / kDnRowsPerItem;
    const int item_bytes = kDnRowsPerItem * f + kDnRowsPerItem * (f / 16);  // qs rows, then their scales
    unsigned char* ring = dn_smem + (size_t)warp * NSTG * item_bytes;
    float4* hs = reinterpret_cast<float4*>(dn_smem + (size_t)NW * NSTG * item_bytes);

    // Offsets were written two kernels back (routing/bucketing) and were
    // complete before gate/up released this grid: Wd can stream at once.
    if (warp == 0)
        build_active(offsets, E, ALLP ? (1 << 30) : tcp, P, s_act, s_beg, s_end, s_cb, &s_n, eslot, nslots);
    __syncthreads();
    int lo, hi;
    item_range(s_cb[s_n] * nq, &lo, &hi);

    auto issue = [&](int i, int st) {
        const int g = i / nq, qd = i - g * nq;
        dn_issue_item(ring + (size_t)st * item_bytes, dqs, dd,
                      (size_t)s_act[locate(g, s_cb, s_n)] * dm + (size_t)qd * kDnRowsPerItem, f, lane);
    };
    auto compute = [&](int i, int st) {
        const int g = i / nq, qd = i - g * nq;
        const int a = locate(g, s_cb, s_n);
        const int c0 = g - s_cb[a];
        const int pb = ALLP ? s_beg[a] : s_beg[a] + c0 * tcp;
        const int pe = ALLP ? s_end[a] : min(s_end[a], pb + tcp);
        if constexpr (G == kMultiG) {
            const unsigned char* b = ring + (size_t)st * item_bytes;
            if (ALLP) dn_compute_multi<KCH>(b, qd, pb, pe, f, dm, hl, sub, hs, pb, s_ptok + pb, s_pw + pb, fuse, out);
            else dn_compute_multi<KCH>(b, qd, pb, pe, f, dm, hl, sub, hs, 0, s_segtok, s_segw, fuse, out);
        } else {
            dn_compute_item<KCH, G, ALLP>(ring + (size_t)st * item_bytes, qd, pb, pe, f, dm, k, T, hl, sub, hs,
                                          s_ptok, s_pw, pair_tok, pair_slot, wts, fuse, out);
        }
    };

    if (ALLP) {
        // start the weight stream, then wait for gate/up before staging h
        const int first = lo + warp;
        const int n = first < hi ? (hi - first + NW - 1) / NW : 0;
#pragma unroll
        for (int j = 0; j < NSTG - 1; ++j) {
            if (j < n) issue(first + j * NW, j);
            else cp_async_commit();
        }
        pdl_wait();  // gate/up complete: h and the combine target are ready
        pdl_launch_dependents();
        for (int q = threadIdx.x; q < P * f4; q += kThreads) {
            const int p = q / f4, qq = q - p * f4;
            hs[p * kTok4 + stage_idx<LPR>(qq)] = __ldcg(reinterpret_cast<const float4*>(h) + (size_t)p * f4 + qq);
        }
        for (int p = threadIdx.x; p < P; p += kThreads) {
            const int tok = __ldcg(pair_tok + p), sl = __ldcg(pair_slot + p);
            const bool ok = tok >= 0 && tok < T && sl >= 0 && sl < k;
            s_ptok[p] = ok ? tok : -1;
            s_pw[p] = ok ? __ldcg(wts + (size_t)tok * k + sl) : 0.f;
        }
        __syncthreads();
        for (int j = 0; j < n; ++j) {
            const int jn = j + NSTG - 1;
            if (jn < n) issue(first + jn * NW, jn % NSTG);
            else cp_async_commit();
            cp_async_wait<NSTG - 1>();
            __syncwarp();
            compute(first + j * NW, j % NSTG);
            __syncwarp();
        }
    } else {
        pdl_wait();
        pdl_launch_dependents();
        for (int seg = lo; seg < hi;) {
            const int g = seg / nq;
            const int seg_end = min(hi, (g + 1) * nq);
            const int a = locate(g, s_cb, s_n);
            const int pb = s_beg[a] + (g - s_cb[a]) * tcp;
            const int pe = min(s_end[a], pb + tcp);
            __syncthreads();
#pragma unroll 4
            for (int q = threadIdx.x; q < (pe - pb) * f4; q += kThreads) {
                const int jj = q / f4, qq = q - jj * f4;
                hs[jj * kTok4 + stage_idx<LPR>(qq)] =
                    __ldcg(reinterpret_cast<const float4*>(h) + (size_t)(pb + jj) * f4 + qq);
            }
            for (int j = threadIdx.x; j < pe - pb; j += kThreads) {
                const int tok = __ldcg(pair_tok + pb + j), sl = __ldcg(pair_slot + pb + j);
                const bool ok = tok >= 0 && tok < T && sl >= 0 && sl < k;
                s_segtok[j] = ok ? tok : -1;
                s_segw[j] = ok ? __ldcg(wts + (size_t)tok * k + sl) : 0.f;
            }
            __syncthreads();
            warp_stream<NSTG>(seg + warp, seg_end, NW, issue, compute);
            seg = seg_end;
        }
    }
    cp_async_wait<0>();
}

int g_num_sms[64] = {0};

int num_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!g_num_sms[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_num_sms[dev] = n > 0 ? n : 148;
    }
    return g_num_sms[dev];
}

template <typename K, typename... Args>
cudaError_t launch_pdl(K kern, int grid, int threads, size_t smem, cudaStream_t s, Args... args) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

constexpr size_t kSmemCap = 220 * 1024;  // dynamic shared memory per CTA we allow ourselves

template <int KCH, int G, bool ALLTOK, int NW, int NSTG>
cudaError_t gateup_go(const float* x, int T, const moe_layer_w& w, const int32_t* offsets, const int32_t* pair_tok,
                      float* h, float* out_init, int residual, int tca, cudaStream_t s) {
    const int dm = w.d_model;
    const size_t ring = (size_t)NW * NSTG * (2 * dm + 2 * (dm / 16));
    const size_t smem = ring + (size_t)tca * KCH * 4 * 32 * 16;
    if (smem > kSmemCap) return cudaErrorInvalidConfiguration;
    return launch_pdl(gateup_cp_kernel<KCH, G, ALLTOK, NW, NSTG>, num_sms(), NW * 32, smem, s, x, T, dm, w.d_ff,
                      w.E, w.gate.qs, w.gate.d, w.up.qs, w.up.d, offsets, pair_tok, h, out_init, residual, tca,
                      T * w.k, w.expert_slot, weight_slots(w));
}

template <int KCH>
cudaError_t gateup_dispatch(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                            const int32_t* pair_tok, float* h, float* out_init, int residual, cudaStream_t s) {
    const int P = T * w.k;
    const int tca = T <= kMultiG ? T : kMultiG;
    const bool alltok = T <= kMultiG && P <= kMaxStagedPairs;
    // ring: 16 warps x 3 stages of one feature (gate + up rows) when the
    // activations are small, 12 warps otherwise
    if (T == 1 && alltok) return gateup_go<KCH, 1, true, 16, 3>(x, T, w, offsets, pair_tok, h, out_init, residual, tca, s);
    if (T <= 2 && alltok) return gateup_go<KCH, 2, true, 16, 3>(x, T, w, offsets, pair_tok, h, out_init, residual, tca, s);
    // 3+ tokens: items of up to kMultiG pairs (a bucket holds at most T <= 8
    // pairs when every token is staged, else chunks of tca = 8)
    if (alltok)
        return gateup_go<KCH, kMultiG, true, 12, 3>(x, T, w, offsets, pair_tok, h, out_init, residual, tca, s);
    return gateup_go<KCH, kMultiG, false, 12, 3>(x, T, w, offsets, pair_tok, h, out_init, residual, tca, s);
}

template <int KCH, int G, bool ALLP, int NW, int NSTG>
cudaError_t down_go(const float* h, int T, const moe_layer_w& w, const int32_t* offsets, const int32_t* pair_tok,
                    const int32_t* pair_slot, const float* wts, int fuse, float* out, int tcp, cudaStream_t s) {
    const int f = w.d_ff;
    const size_t ring = (size_t)NW * NSTG * (kDnRowsPerItem * f + kDnRowsPerItem * (f / 16));
    const size_t smem = ring + (size_t)tcp * KCH * 4 * 16 * 16;
    if (smem > kSmemCap) return cudaErrorInvalidConfiguration;
    return launch_pdl(down_cp_kernel<KCH, G, ALLP, NW, NSTG>, num_sms(), NW * 32, smem, s, h, T, f, w.d_model, w.E,
                      w.k, w.down.qs, w.down.d, offsets, pair_tok, pair_slot, wts, fuse, out, tcp, w.expert_slot,
                      weight_slots(w));
}

template <int KCH>
cudaError_t down_dispatch(const float* h, int T, const moe_layer_w& w, const int32_t* offsets,
                          const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse, float* out,
                          cudaStream_t s) {
    const int P = T * w.k;
    const size_t tok_bytes = (size_t)KCH * 4 * 16 * 16;
    const bool allp = (size_t)P * tok_bytes <= 48 * 1024 && P <= kMaxStagedPairs;
    if (T == 1 && allp)
        return down_go<KCH, 1, true, 16, 3>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, P, s);
    if (T <= 2 && allp) return down_go<KCH, 4, true, 16, 3>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, P, s);
    // 3+ tokens: items of up to kMultiG pairs (whole buckets of <= T <= 8
    // pairs when every pair's h is staged, else chunks of tcp = kMultiG)
    if (allp && T <= kMultiG)
        return down_go<KCH, kMultiG, true, 16, 3>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, P, s);
    return down_go<KCH, kMultiG, false, 16, 3>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, kMultiG, s);
}

}  // namespace

// Whether both kernels' shared memory (rings + staged activations), in the
// configuration the dispatch above picks for T tokens, fits the cap.
bool ffn_stream_fits(const moe_layer_w& w, int T) {
    const int dm = w.d_model, f = w.d_ff, P = T * w.k;
    const int kg = (dm / 16 + 31) / 32, KCHg = kg <= 2 ? kg : 4;
    const int kd = (f / 16 + 15) / 16, KCHd = kd <= 3 ? kd : 4;
    const int tca = T <= kMultiG ? T : kMultiG;
    const bool alltok = T <= kMultiG && P <= kMaxStagedPairs;
    const int nwg = (T <= 2 && alltok) ? 16 : 12;
    const size_t gu = (size_t)nwg * 3 * (2 * dm + 2 * (dm / 16)) + (size_t)tca * KCHg * 4 * 32 * 16;
    const size_t tok_bytes = (size_t)KCHd * 4 * 16 * 16;
    const bool allp = (size_t)P * tok_bytes <= 48 * 1024 && P <= kMaxStagedPairs;
    const int tcp = (allp && (T <= 2 || T <= kMultiG)) ? P : kMultiG;
    const size_t dn = (size_t)16 * 3 * (kDnRowsPerItem * f + kDnRowsPerItem * (f / 16)) + (size_t)tcp * tok_bytes;
    return gu <= kSmemCap && dn <= kSmemCap;
}

bool ffn_stream_supported(const moe_layer_w& w) {
    // whole 16-byte pieces of weights and of each row's scales: K % 256 == 0;
    // down items are 4 whole rows; at most 4 chunks per lane.
    return w.wfmt == MOE_WFMT_Q8_0 && w.d_model % 256 == 0 && w.d_ff % 256 == 0 && w.d_model % kDnRowsPerItem == 0 && w.d_model <= 2048 &&
           w.d_ff <= 1024;
}

cudaError_t launch_ffn_stream(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                              const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse_combine,
                              float* out_or_ypairs, int residual, float* h, int32_t* status, cudaStream_t s) {
    (void)status;
    if (T == 0) return cudaSuccess;
    float* out_init = fuse_combine ? out_or_ypairs : nullptr;
    const int kg = (w.d_model / 16 + 31) / 32;
    cudaError_t err;
    switch (kg) {
        case 1: err = gateup_dispatch<1>(x, T, w, offsets, pair_tok, h, out_init, residual, s); break;
        case 2: err = gateup_dispatch<2>(x, T, w, offsets, pair_tok, h, out_init, residual, s); break;
        default: err = gateup_dispatch<4>(x, T, w, offsets, pair_tok, h, out_init, residual, s); break;
    }
    if (err != cudaSuccess) return err;
    const int kd = (w.d_ff / 16 + 15) / 16;
    switch (kd) {
        case 1: return down_dispatch<1>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs, s);
        case 2: return down_dispatch<2>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs, s);
        case 3: return down_dispatch<3>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs, s);
        default: return down_dispatch<4>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs, s);
    }
}

}  // namespace moe
