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
// contiguous range of weight tiles (one expert, RB consecutive rows; the rows
// of one expert matrix are contiguous, so a tile is one contiguous run of
// int8 plus one run of fp16 scales).  One producer thread streams tiles into
// a ring of shared-memory stages with 1-D bulk copies (cp.async.bulk,
// completion on an mbarrier), keeping up to S tiles (~100 KB) in flight per
// SM; eight consumer warps each take one row of the landed tile into
// registers, release the stage, and contract it with the staged activations
// of every token routed to that expert.  Each weight byte is read from HBM
// once per layer.  The down kernel is launched as a programmatic dependent of
// gate/up: its producer starts streaming Wd while gate/up finishes, and only
// its consumers wait for h.
#include "common.cuh"
#include "pipeline.cuh"

namespace moe {

namespace {

constexpr int kCW = 8;                      // consumer warps
constexpr int kStreamThreads = (kCW + 1) * 32;
constexpr int kGuRows = kCW;                // gate/up tile: 8 output features (8 gate + 8 up rows)
constexpr int kDnRows = 2 * kCW;            // down tile: 16 rows, 16 lanes per row

template <int LPR>
__device__ __forceinline__ int stage_idx(int q) {
    const int c = q >> 2, m = q & 3;
    return ((c / LPR) * 4 + m) * LPR + (c % LPR);
}

// Active experts (non-empty buckets) in id order, by warp 0, and the work
// list they imply: expert a's bucket is cut into chunks of at most `chunk`
// pairs (the activations one pass stages in shared memory); s_cb[a] is the
// index of a's first chunk and s_cb[n] the total.  Offsets are read through
// L2 (written by an earlier kernel of this layer).
__device__ void build_active(const int32_t* offsets, int E, int chunk, int* s_act, int* s_beg, int* s_end,
                             int* s_cb, int* s_n) {
    const int lane = threadIdx.x & 31;
    int n = 0, nc = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int lo = e < E ? __ldcg(offsets + e) : 0;
        const int hi = e < E ? __ldcg(offsets + e + 1) : 0;
        const bool a = hi > lo;
        const uint32_t m = __ballot_sync(0xffffffffu, a);
        const int my_c = a ? (hi - lo + chunk - 1) / chunk : 0;
        int incl = my_c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (a) {
            const int j = n + __popc(m & ((1u << lane) - 1u));
            s_act[j] = e;
            s_beg[j] = lo;
            s_end[j] = hi;
            s_cb[j] = nc + incl - my_c;
        }
        n += __popc(m);
        nc += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
        *s_n = n;
        s_cb[n] = nc;
    }
}

// Work item -> (active expert a, chunk c of its bucket, row block rb).
__device__ __forceinline__ void decode_item(int i, int nrb, const int* s_cb, int n, int* a, int* c, int* rb) {
    const int g = i / nrb;
    *rb = i - g * nrb;
    int lo = 0, hi = n - 1;  // largest a with s_cb[a] <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_cb[mid] <= g) lo = mid;
        else hi = mid - 1;
    }
    *a = lo;
    *c = g - s_cb[lo];
}

__device__ __forceinline__ void tile_range(int n_tiles, int* lo, int* hi) {
    const long long b = blockIdx.x, G = gridDim.x;
    *lo = (int)(b * n_tiles / G);
    *hi = (int)((b + 1) * n_tiles / G);
}

// ============================================================== gate / up ==
// KCH: 16-byte chunks per lane (d_model / 512, rounded up); G: tokens per
// register block; ALLTOK: all T tokens' x staged once (T <= tca) instead of
// per-expert bucket chunks.
template <int KCH, int G, bool ALLTOK>
__global__ void __launch_bounds__(kStreamThreads, 1) gateup_stream_kernel(
    const float* __restrict__ x, int T, int dm, int f, int E, const int8_t* __restrict__ gqs,
    const uint16_t* __restrict__ gd, const int8_t* __restrict__ uqs, const uint16_t* __restrict__ ud,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_tok, float* __restrict__ h,
    float* __restrict__ out_init, int init_residual, int S, int tca, int32_t* status) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_act[MOE_MAX_EXPERTS], s_beg[MOE_MAX_EXPERTS], s_end[MOE_MAX_EXPERTS];
    __shared__ int s_cb[MOE_MAX_EXPERTS + 1], s_n;
    constexpr int kTok4 = KCH * 4 * 32;  // float4 per staged token
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = dm / 16;
    const uint32_t qbytes = (uint32_t)kGuRows * dm;        // one matrix's qs per tile
    const uint32_t sbytes = (uint32_t)kGuRows * dm / 16;   // one matrix's scales per tile
    const uint32_t stage_bytes = 2 * qbytes + 2 * sbytes;
    float4* xs = reinterpret_cast<float4*>(smem + (size_t)S * stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * stage_bytes + (size_t)tca * kTok4 * 16);
    uint64_t* empty = full + S;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kCW);
        }
        fence_barrier_init();
    }
    pdl_wait();  // routing / bucketing of this layer complete and visible
    if (warp == 0) build_active(offsets, E, ALLTOK ? (1 << 30) : tca, s_act, s_beg, s_end, s_cb, &s_n);
    if (out_init) {  // combine target: (residual ? x : 0), consumed by the down kernel
        const size_t n4 = (size_t)T * dm / 4;
        float4* o4 = reinterpret_cast<float4*>(out_init);
        const float4* x4 = reinterpret_cast<const float4*>(x);
        for (size_t i = (size_t)blockIdx.x * kStreamThreads + threadIdx.x; i < n4;
             i += (size_t)gridDim.x * kStreamThreads)
            o4[i] = init_residual ? __ldcg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (ALLTOK) {
        const int d4 = dm / 4;
        for (int i = threadIdx.x; i < T * d4; i += kStreamThreads) {
            const int t = i / d4, q = i - t * d4;
            xs[t * kTok4 + stage_idx<32>(q)] = __ldcg(reinterpret_cast<const float4*>(x) + (size_t)t * d4 + q);
        }
    }
    __syncthreads();
    pdl_launch_dependents();
    const int nrb = f / kGuRows;
    const int n_tiles = s_cb[s_n] * nrb;
    int lo, hi;
    tile_range(n_tiles, &lo, &hi);

    if (warp == kCW) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int i = lo, j = 0; i < hi; ++i, ++j) {
                const int s = j % S;
                if (j >= S && !mbar_wait(empty + s, ((j / S) - 1) & 1)) {
                    flag_status(status, MOE_STATUS_TIMEOUT_BIT);
                    break;
                }
                int a, c, rb;
                decode_item(i, nrb, s_cb, s_n, &a, &c, &rb);
                const size_t row = (size_t)s_act[a] * f + (size_t)rb * kGuRows;
                unsigned char* st = smem + (size_t)s * stage_bytes;
                mbar_arrive_expect_tx(full + s, stage_bytes);
                bulk_g2s_stream(st, gqs + row * dm, qbytes, full + s, pol);
                bulk_g2s_stream(st + qbytes, uqs + row * dm, qbytes, full + s, pol);
                bulk_g2s_stream(st + 2 * qbytes, gd + row * (dm / 32), sbytes, full + s, pol);
                bulk_g2s_stream(st + 2 * qbytes + sbytes, ud + row * (dm / 32), sbytes, full + s, pol);
            }
            // drain: every issued copy has landed before the CTA may exit
            for (int i = (hi - lo > S ? hi - S : lo); i < hi; ++i) {
                const int j = i - lo;
                mbar_wait(full + (j % S), (j / S) & 1);
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    int staged = -1;  // work chunk (index into s_cb numbering) whose activations are in xs
    bool dead = false;
    for (int i = lo, j = 0; i < hi; ++i, ++j) {
        const int s = j % S;
        int a, c, rb;
        decode_item(i, nrb, s_cb, s_n, &a, &c, &rb);
        const int r = rb * kGuRows + warp;
        if (!dead && !mbar_wait(full + s, (j / S) & 1)) {
            // keep walking the same schedule (the consumers' named barriers
            // must stay matched); the status word marks the output invalid
            flag_status(status, MOE_STATUS_TIMEOUT_BIT);
            dead = true;
        }
        const unsigned char* st = smem + (size_t)s * stage_bytes;
        uint4 gq[KCH], uq[KCH];
        float gs[KCH], us[KCH];
#pragma unroll
        for (int c4 = 0; c4 < KCH; ++c4) {
            const int c = lane + 32 * c4;
            if (c < nch) {
                gq[c4] = *reinterpret_cast<const uint4*>(st + (size_t)warp * dm + c * 16);
                uq[c4] = *reinterpret_cast<const uint4*>(st + qbytes + (size_t)warp * dm + c * 16);
                const __half* gsc = reinterpret_cast<const __half*>(st + 2 * qbytes);
                const __half* usc = reinterpret_cast<const __half*>(st + 2 * qbytes + sbytes);
                gs[c4] = __half2float(gsc[warp * (dm / 32) + (c >> 1)]);
                us[c4] = __half2float(usc[warp * (dm / 32) + (c >> 1)]);
            } else {
                gq[c4] = make_uint4(0, 0, 0, 0);
                uq[c4] = make_uint4(0, 0, 0, 0);
                gs[c4] = 0.f;
                us[c4] = 0.f;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + s);

        const int pb = ALLTOK ? s_beg[a] : s_beg[a] + c * tca;
        const int pe = ALLTOK ? s_end[a] : min(s_end[a], pb + tca);
        {
            if (!ALLTOK && s_cb[a] + c != staged) {
                named_bar(1, kCW * 32);  // everyone done with the previous chunk
                const int d4 = dm / 4;
                for (int q = threadIdx.x; q < (pe - pb) * d4; q += kCW * 32) {
                    const int jj = q / d4, qq = q - jj * d4;
                    const int t = __ldcg(pair_tok + pb + jj);
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (t >= 0 && t < T) v = __ldcg(reinterpret_cast<const float4*>(x) + (size_t)t * d4 + qq);
                    xs[jj * kTok4 + stage_idx<32>(qq)] = v;
                }
                named_bar(1, kCW * 32);
                staged = s_cb[a] + c;
            }
            for (int pp = pb; pp < pe; pp += G) {
                const int ng = min(G, pe - pp);
                int toff[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    int o = 0;
                    if (g < ng) {
                        if (ALLTOK) {
                            int t = __ldcg(pair_tok + pp + g);
                            t = (t >= 0 && t < T) ? t : 0;
                            o = t * kTok4;
                        } else {
                            o = (pp + g - pb) * kTok4;
                        }
                    }
                    toff[g] = o;
                }
                float ga[G], ua[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    ga[g] = 0.f;
                    ua[g] = 0.f;
                }
#pragma unroll
                for (int c4 = 0; c4 < KCH; ++c4) {
                    if (lane + 32 * c4 < nch) {
                        float gp[G], up[G];
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            gp[g] = 0.f;
                            up[g] = 0.f;
                        }
                        const uint32_t gw[4] = {gq[c4].x, gq[c4].y, gq[c4].z, gq[c4].w};
                        const uint32_t uw[4] = {uq[c4].x, uq[c4].y, uq[c4].z, uq[c4].w};
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float4 gf = i8x4_to_f32x4(gw[m]);
                            const float4 uf = i8x4_to_f32x4(uw[m]);
#pragma unroll
                            for (int g = 0; g < G; ++g) {
                                if (g < ng) {
                                    const float4 xv = xs[toff[g] + (c4 * 4 + m) * 32 + lane];
                                    gp[g] = dot4(gf, xv, gp[g]);
                                    up[g] = dot4(uf, xv, up[g]);
                                }
                            }
                        }
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            ga[g] = fmaf(gs[c4], gp[g], ga[g]);
                            ua[g] = fmaf(us[c4], up[g], ua[g]);
                        }
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    ga[g] = warp_sum(ga[g]);
                    ua[g] = warp_sum(ua[g]);
                }
#pragma unroll
                for (int g = 0; g < G; ++g)
                    if (lane == g && g < ng) h[(size_t)(pp + g) * f + r] = silu_f(ga[g]) * ua[g];
            }
        }
    }
}

// =================================================================== down ==
// 16 lanes per row, two rows per consumer warp, KCH 16-byte chunks per lane
// (d_ff / 256, rounded up).  ALLP: all P pairs' h staged once.
template <int KCH, int G, bool ALLP>
__global__ void __launch_bounds__(kStreamThreads, 1) down_stream_kernel(
    const float* __restrict__ h, int T, int f, int dm, int E, int k, const int8_t* __restrict__ dqs,
    const uint16_t* __restrict__ dd, const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_tok,
    const int32_t* __restrict__ pair_slot, const float* __restrict__ wts, int fuse, float* __restrict__ out, int S,
    int tcp, int32_t* status) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_act[MOE_MAX_EXPERTS], s_beg[MOE_MAX_EXPERTS], s_end[MOE_MAX_EXPERTS];
    __shared__ int s_cb[MOE_MAX_EXPERTS + 1], s_n;
    constexpr int LPR = 16;
    constexpr int kTok4 = KCH * 4 * LPR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hl = lane & 15, sub = lane >> 4;
    const int nch = f / 16;
    const uint32_t qbytes = (uint32_t)kDnRows * f;
    const uint32_t sbytes = (uint32_t)kDnRows * f / 16;
    const uint32_t stage_bytes = qbytes + sbytes;
    float4* hs = reinterpret_cast<float4*>(smem + (size_t)S * stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * stage_bytes + (size_t)tcp * kTok4 * 16);
    uint64_t* empty = full + S;
    const int P = T * k;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kCW);
        }
        fence_barrier_init();
    }
    // Offsets were written two kernels back (routing/bucketing), complete
    // before gate/up released this grid, so the weight stream can start now.
    if (warp == 0) build_active(offsets, E, ALLP ? (1 << 30) : tcp, s_act, s_beg, s_end, s_cb, &s_n);
    __syncthreads();
    const int nrb = dm / kDnRows;
    const int n_tiles = s_cb[s_n] * nrb;
    int lo, hi;
    tile_range(n_tiles, &lo, &hi);

    if (warp == kCW) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int i = lo, j = 0; i < hi; ++i, ++j) {
                const int s = j % S;
                if (j >= S && !mbar_wait(empty + s, ((j / S) - 1) & 1)) {
                    flag_status(status, MOE_STATUS_TIMEOUT_BIT);
                    break;
                }
                int a, c, rb;
                decode_item(i, nrb, s_cb, s_n, &a, &c, &rb);
                const size_t row = (size_t)s_act[a] * dm + (size_t)rb * kDnRows;
                unsigned char* st = smem + (size_t)s * stage_bytes;
                mbar_arrive_expect_tx(full + s, stage_bytes);
                bulk_g2s_stream(st, dqs + row * f, qbytes, full + s, pol);
                bulk_g2s_stream(st + qbytes, dd + row * (f / 32), sbytes, full + s, pol);
            }
            for (int i = (hi - lo > S ? hi - S : lo); i < hi; ++i) {
                const int j = i - lo;
                mbar_wait(full + (j % S), (j / S) & 1);
            }
        }
        return;
    }

    pdl_wait();  // gate/up complete: h and the combine target are ready
    pdl_launch_dependents();
    const int f4 = f / 4;
    if (ALLP) {
        for (int q = threadIdx.x; q < P * f4; q += kCW * 32) {
            const int p = q / f4, qq = q - p * f4;
            hs[p * kTok4 + stage_idx<LPR>(qq)] = __ldcg(reinterpret_cast<const float4*>(h) + (size_t)p * f4 + qq);
        }
        named_bar(1, kCW * 32);
    }
    int staged = -1;
    bool dead = false;
    for (int i = lo, j = 0; i < hi; ++i, ++j) {
        const int s = j % S;
        int a, c, rb;
        decode_item(i, nrb, s_cb, s_n, &a, &c, &rb);
        const int rl = warp * 2 + sub;  // row within the tile
        const int o = rb * kDnRows + rl;
        if (!dead && !mbar_wait(full + s, (j / S) & 1)) {
            flag_status(status, MOE_STATUS_TIMEOUT_BIT);
            dead = true;
        }
        const unsigned char* st = smem + (size_t)s * stage_bytes;
        uint4 wq[KCH];
        float wsc[KCH];
#pragma unroll
        for (int c4 = 0; c4 < KCH; ++c4) {
            const int c = hl + LPR * c4;
            if (c < nch) {
                wq[c4] = *reinterpret_cast<const uint4*>(st + (size_t)rl * f + c * 16);
                wsc[c4] = __half2float(reinterpret_cast<const __half*>(st + qbytes)[rl * (f / 32) + (c >> 1)]);
            } else {
                wq[c4] = make_uint4(0, 0, 0, 0);
                wsc[c4] = 0.f;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + s);

        const int pb = ALLP ? s_beg[a] : s_beg[a] + c * tcp;
        const int pe = ALLP ? s_end[a] : min(s_end[a], pb + tcp);
        {
            if (!ALLP && s_cb[a] + c != staged) {
                named_bar(1, kCW * 32);
                for (int q = threadIdx.x; q < (pe - pb) * f4; q += kCW * 32) {
                    const int jj = q / f4, qq = q - jj * f4;
                    hs[jj * kTok4 + stage_idx<LPR>(qq)] =
                        __ldcg(reinterpret_cast<const float4*>(h) + (size_t)(pb + jj) * f4 + qq);
                }
                named_bar(1, kCW * 32);
                staged = s_cb[a] + c;
            }
            for (int pp = pb; pp < pe; pp += G) {
                const int ng = min(G, pe - pp);
                int hoff[G];
#pragma unroll
                for (int g = 0; g < G; ++g) hoff[g] = (g < ng ? (ALLP ? (pp + g) : (pp + g - pb)) : 0) * kTok4;
                float acc[G];
#pragma unroll
                for (int g = 0; g < G; ++g) acc[g] = 0.f;
#pragma unroll
                for (int c4 = 0; c4 < KCH; ++c4) {
                    if (hl + LPR * c4 < nch) {
                        float part[G];
#pragma unroll
                        for (int g = 0; g < G; ++g) part[g] = 0.f;
                        const uint32_t ww[4] = {wq[c4].x, wq[c4].y, wq[c4].z, wq[c4].w};
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float4 wf = i8x4_to_f32x4(ww[m]);
#pragma unroll
                            for (int g = 0; g < G; ++g)
                                if (g < ng) part[g] = dot4(wf, hs[hoff[g] + (c4 * 4 + m) * LPR + hl], part[g]);
                        }
#pragma unroll
                        for (int g = 0; g < G; ++g) acc[g] = fmaf(wsc[c4], part[g], acc[g]);
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) acc[g] = group_sum<LPR>(acc[g]);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (hl == g && g < ng) {
                        const int p = pp + g;
                        if (fuse) {
                            const int tok = __ldcg(pair_tok + p), sl = __ldcg(pair_slot + p);
                            if (tok >= 0 && tok < T && sl >= 0 && sl < k)
                                atomicAdd(out + (size_t)tok * dm + o, __ldcg(wts + (size_t)tok * k + sl) * acc[g]);
                        } else {
                            out[(size_t)p * dm + o] = acc[g];
                        }
                    }
                }
            }
        }
    }
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
cudaError_t launch_pdl(K kern, int grid, size_t smem, cudaStream_t s, Args... args) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kStreamThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

constexpr size_t kGuSmemBudget = 120 * 1024;  // leaves room for a co-resident down CTA
constexpr size_t kDnSmemBudget = 96 * 1024;

template <int KCH>
cudaError_t gateup_dispatch(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                            const int32_t* pair_tok, float* h, float* out_init, int residual, int32_t* status,
                            cudaStream_t s) {
    const int dm = w.d_model;
    const size_t stage = 2 * (size_t)kGuRows * dm + 2 * (size_t)kGuRows * dm / 16;
    const size_t tok_bytes = (size_t)KCH * 4 * 32 * 16;
    int tca = T <= 8 ? T : 8;
    while (tca > 1 && (size_t)tca * tok_bytes > 64 * 1024) --tca;
    const long long avail = (long long)kGuSmemBudget - (long long)tca * (long long)tok_bytes;
    int S = (int)(avail / (long long)(stage + 16));
    if (S > 6) S = 6;
    if (S < 2) S = 2;
    const size_t smem = (size_t)S * stage + (size_t)tca * tok_bytes + (size_t)2 * S * 8;
    if (smem > 200 * 1024) return cudaErrorInvalidConfiguration;
    const int grid = num_sms();
    if (T == 1)
        return launch_pdl(gateup_stream_kernel<KCH, 1, true>, grid, smem, s, x, T, dm, w.d_ff, w.E, w.gate.qs,
                          w.gate.d, w.up.qs, w.up.d, offsets, pair_tok, h, out_init, residual, S, tca, status);
    if (T <= tca)
        return launch_pdl(gateup_stream_kernel<KCH, 4, true>, grid, smem, s, x, T, dm, w.d_ff, w.E, w.gate.qs,
                          w.gate.d, w.up.qs, w.up.d, offsets, pair_tok, h, out_init, residual, S, tca, status);
    return launch_pdl(gateup_stream_kernel<KCH, 4, false>, grid, smem, s, x, T, dm, w.d_ff, w.E, w.gate.qs,
                      w.gate.d, w.up.qs, w.up.d, offsets, pair_tok, h, out_init, residual, S, tca, status);
}

template <int KCH>
cudaError_t down_dispatch(const float* h, int T, const moe_layer_w& w, const int32_t* offsets,
                          const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse, float* out,
                          int32_t* status, cudaStream_t s) {
    const int f = w.d_ff;
    const int P = T * w.k;
    const size_t stage = (size_t)kDnRows * f + (size_t)kDnRows * f / 16;
    const size_t tok_bytes = (size_t)KCH * 4 * 16 * 16;
    const bool allp = (size_t)P * tok_bytes <= 48 * 1024;
    const int tcp = allp ? P : 8;
    int S = (int)(((long long)kDnSmemBudget - (long long)tcp * (long long)tok_bytes) / (long long)(stage + 16));
    if (S > 8) S = 8;
    if (S < 2) S = 2;
    const size_t smem = (size_t)S * stage + (size_t)tcp * tok_bytes + (size_t)2 * S * 8;
    const int grid = num_sms();
    if (T == 1)
        return launch_pdl(down_stream_kernel<KCH, 1, true>, grid, smem, s, h, T, f, w.d_model, w.E, w.k, w.down.qs,
                          w.down.d, offsets, pair_tok, pair_slot, wts, fuse, out, S, tcp, status);
    if (allp)
        return launch_pdl(down_stream_kernel<KCH, 4, true>, grid, smem, s, h, T, f, w.d_model, w.E, w.k, w.down.qs,
                          w.down.d, offsets, pair_tok, pair_slot, wts, fuse, out, S, tcp, status);
    return launch_pdl(down_stream_kernel<KCH, 4, false>, grid, smem, s, h, T, f, w.d_model, w.E, w.k, w.down.qs,
                      w.down.d, offsets, pair_tok, pair_slot, wts, fuse, out, S, tcp, status);
}

}  // namespace

bool ffn_stream_supported(const moe_layer_w& w) {
    // tile = 8 (gate/up) or 16 (down) whole rows: 16-byte aligned runs of qs
    // and scales need K % 64 == 0; rows must fill whole tiles.
    return w.d_model % 64 == 0 && w.d_ff % 64 == 0 && w.d_ff % kGuRows == 0 && w.d_model % kDnRows == 0 &&
           w.d_model <= 4096 && w.d_ff <= 1024;
}

cudaError_t launch_ffn_stream(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                              const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse_combine,
                              float* out_or_ypairs, int residual, float* h, int32_t* status, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    float* out_init = fuse_combine ? out_or_ypairs : nullptr;
    const int kg = (w.d_model / 16 + 31) / 32;
    cudaError_t err;
    switch (kg) {
        case 1: err = gateup_dispatch<1>(x, T, w, offsets, pair_tok, h, out_init, residual, status, s); break;
        case 2: err = gateup_dispatch<2>(x, T, w, offsets, pair_tok, h, out_init, residual, status, s); break;
        case 3:
        case 4: err = gateup_dispatch<4>(x, T, w, offsets, pair_tok, h, out_init, residual, status, s); break;
        default: err = gateup_dispatch<8>(x, T, w, offsets, pair_tok, h, out_init, residual, status, s); break;
    }
    if (err != cudaSuccess) return err;
    const int kd = (w.d_ff / 16 + 15) / 16;
    switch (kd) {
        case 1: return down_dispatch<1>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs,
                                        status, s);
        case 2: return down_dispatch<2>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs,
                                        status, s);
        case 3: return down_dispatch<3>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs,
                                        status, s);
        default: return down_dispatch<4>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs,
                                         status, s);
    }
}

}  // namespace moe
