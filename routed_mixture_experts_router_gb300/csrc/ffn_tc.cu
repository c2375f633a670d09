// Expert SwiGLU FFNs on the tcgen05 tensor cores (the prefill path): bf16
// operands, fp32 accumulation in TMEM, Q8_0 dequantisation fused into the
// operand staging, SwiGLU fused into the gate/up epilogue and the weighted
// combine fused into the down epilogue.
//
//   gather   xb[p] = bf16(x[token(p)])                      pairs in bucket order
//   gate/up  h[p][r] = bf16( silu(Wg_e[r] . xb[p]) * (Wu_e[r] . xb[p]) )
//   down     out[t][o] += w[t][slot] * (Wd_e[o] . h[p])     (or ypairs[p][o])
// Q8_0 weights w = q * d (amalgafy.com/technical-overview, "Validated GPU
// foundation"); down projection K=768 -> 2048 rows and prefill batches of
// 768 / 1024 tokens (expxa.com reuse-ordering-qualification, "What changed
// from the first experiment"); activations cast for the expert contraction
// ("including routing and quantization", same page, "Operator gains ...").
//
// Design (one persistent 640-thread CTA per SM).  A work unit is one expert,
// one 128-row tile of its weight matrix (the MMA M dimension: "swap AB", so
// the small, ragged token count is N) and up to 128 of its tokens (N, padded
// to a multiple of 16).  Warp roles:
//   warp 0       TMA producer: int8 weight tiles (128 rows x 128 K, 128-byte
//                swizzle) into a raw ring
//   warp 2       TMA producer: bf16 token tiles (N x 64 K) into the operand
//                ring (separate, so the weight stream never waits on it)
//   warp 1       MMA issuer (one thread): tcgen05.mma kind::f16, M=128,
//                K=16 per instruction, A from TMEM, B from shared memory,
//                into TMEM accumulators (double-buffered for the down
//                projection, single for gate/up, whose two matrices fill
//                the columns the A stages leave)
//   warps 4-11   dequantisation: thread = (row, half of each 64-K operand
//                stage); int8 -> fp32 exactly, times the block's fp16 scale,
//                -> bf16 (RNE), stored straight into TMEM (lane = weight row,
//                its warp's lane quadrant) as the MMA's A operand: no
//                shared-memory round trip for the dequantised weights
//   warps 12-19  epilogue (two per TMEM lane quadrant, alternate 16-token
//                column chunks): tcgen05.ld of the accumulator (lane = row),
//                SwiGLU -> bf16 h, or the weighted combine into out
// Every mbarrier wait is bounded: past the deadline the CTA flags
// MOE_STATUS_TIMEOUT in the status word and stops; all copies and MMAs it
// started are drained before TMEM is freed.
#include <atomic>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "pipeline.cuh"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int kTcThreads = 640;  // 4 control warps, 8 dequantisation warps, 8 epilogue warps
constexpr int kBM = 128;      // weight rows per unit (MMA M)
constexpr int kBKR = 128;     // bytes of a weight row per raw stage (128 K of Q8_0, 256 K of Q4_0)
constexpr int kBK = 64;       // bf16 K per operand stage (one 128-byte row)
constexpr int kBN = 128;      // max tokens per unit (MMA N)
constexpr int kReuseBand = 4;  // row tiles per band of the reuse-ordering traversal (down projection)
constexpr int kBRows = 32;    // token rows per TMA box
// Ring depths.  The raw (int8) ring is what keeps HBM busy: at a few
// microseconds of loaded latency a sustained ~45 GB/s per SM needs ~100 KB of
// weights in flight per SM, so shared memory goes to raw stages first and the
// operand (bf16) ring keeps only the depth the dequant -> MMA hand-off needs.
template <int NMAT>
struct TcRing {
    static constexpr int RS = NMAT == 2 ? 4 : 6;  // raw stages (NMAT x (16 KB + 2 KB scales), shared memory)
    static constexpr int AS = 4;                  // operand stages: NMAT bf16 A tiles in TMEM + one B tile
    static constexpr int NBUF = NMAT == 2 ? 1 : 2;  // accumulator buffers (TMEM)
    static constexpr uint32_t ACC_COLS = NMAT * kBN * NBUF;
    static constexpr uint32_t A_COLS = kBK / 2;   // one bf16 A tile (128 rows x 64 K): 32 columns
    static_assert(ACC_COLS + AS * NMAT * A_COLS <= 512, "TMEM budget");
};
constexpr int kTile = 16384;  // one 128 x 128-byte tile
constexpr int kScTile = 2048;  // scales of one raw stage: 128 rows x 8 fp16 (a 16-byte aligned window)
constexpr int kDqWarp0 = 4, kDqWarps = 8, kEpWarp0 = 12, kEpWarps = 8;
constexpr int kCpt = 4 / (kDqWarps / 4);  // 16-K chunks per dequantisation thread and operand stage
static_assert(kCpt == 2, "a dequantisation thread covers one 32-wide block of an operand stage");

struct TcParams {
    int K;     // reduction length (d_model for gate/up, d_ff for down)
    int rows;  // weight rows per expert (d_ff for gate/up, d_model for down)
    int E, T, k;
    const int32_t* offsets;
    const int32_t* pair_tok;
    const int32_t* pair_slot;
    const float* wts;
    const uint16_t* d0;  // fp16 scales of matrix 0 (gate or down)
    const uint16_t* d1;  // fp16 scales of matrix 1 (up) or null
    __nv_bfloat16* h;    // EPI 0: h [P][rows]
    float* out;          // EPI 1: out [T][rows] (+=); EPI 2: ypairs [P][rows]
    int32_t* status;
    const int32_t* eslot;  // expert -> arena slot, or null (weights in expert order)
    int nslots;
    int band;              // unit order: 0 chunk-major, > 0 bands of that many row tiles (rows / kBM % band == 0)
};

typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_pack(float a, float b) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(f32x2 v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
// two fp32 -> bf16x2 (round to nearest even); `lo` lands in the low half
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// 16 unsigned bytes u (one 16-byte word) -> 16 bf16 (two 16-byte words),
// each w = (u - c0) * d computed exactly in fp32 and then rounded to bf16
// (RNE); cc = -(32768 + c0) * d.  The byte is placed in bits 8..15 of the
// float 2^15, giving v = 32768 + u exactly; one FMA v * d + cc then yields
// (u - c0) * d.  The exact result has at most 19 significant bits (an 8-bit
// integer times an 11-bit fp16 value) and cc is exact too (a 13-bit integer
// times d), so the FMA's single rounding changes nothing.
// Q8_0: u = q + 128 (c0 = 128); Q4_0: u = the nibble n (c0 = 8).
__device__ __forceinline__ void dequant16_u(const uint32_t (&w)[4], f32x2 dd, f32x2 cc, uint4& o0, uint4& o1) {
    uint32_t r[8];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint32_t u = w[m];
        const f32x2 lo = f2_fma(f2_pack(__uint_as_float(__byte_perm(u, 0x47000000u, 0x7504)),
                                        __uint_as_float(__byte_perm(u, 0x47000000u, 0x7514))),
                                dd, cc);
        const f32x2 hi = f2_fma(f2_pack(__uint_as_float(__byte_perm(u, 0x47000000u, 0x7524)),
                                        __uint_as_float(__byte_perm(u, 0x47000000u, 0x7534))),
                                dd, cc);
        float a, b, c, e;
        f2_unpack(lo, a, b);
        f2_unpack(hi, c, e);
        r[2 * m] = bf16x2_rn(a, b);
        r[2 * m + 1] = bf16x2_rn(c, e);
    }
    o0 = make_uint4(r[0], r[1], r[2], r[3]);
    o1 = make_uint4(r[4], r[5], r[6], r[7]);
}

// Q8_0: 16 values of one block (one 16-byte word of the device layout: bytes u = q + 128).
__device__ __forceinline__ void dequant16(uint4 q, f32x2 dd, f32x2 cc, uint4& o0, uint4& o1) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};  // bytes u = q + 128 (device layout)
    dequant16_u(w, dd, cc, o0, o1);
}

// Q4_0: one whole block (16 bytes of nibbles, byte j = element j in its low
// nibble and element j + 16 in its high nibble) -> its 32 values in order:
// v[0..7] elements 0..15, v[8..15] elements 16..31.
__device__ __forceinline__ void dequant32_q4(uint4 q, f32x2 dd, f32x2 cc, uint32_t* v) {
    const uint32_t lo[4] = {q.x & 0x0F0F0F0Fu, q.y & 0x0F0F0F0Fu, q.z & 0x0F0F0F0Fu, q.w & 0x0F0F0F0Fu};
    const uint32_t hi[4] = {(q.x >> 4) & 0x0F0F0F0Fu, (q.y >> 4) & 0x0F0F0F0Fu, (q.z >> 4) & 0x0F0F0F0Fu,
                            (q.w >> 4) & 0x0F0F0F0Fu};
    uint4 a0, a1, b0, b1;
    dequant16_u(lo, dd, cc, a0, a1);
    dequant16_u(hi, dd, cc, b0, b1);
    v[0] = a0.x, v[1] = a0.y, v[2] = a0.z, v[3] = a0.w, v[4] = a1.x, v[5] = a1.y, v[6] = a1.z, v[7] = a1.w;
    v[8] = b0.x, v[9] = b0.y, v[10] = b0.z, v[11] = b0.w, v[12] = b1.x, v[13] = b1.y, v[14] = b1.z, v[15] = b1.w;
}

// silu(g) * u for the bf16 h of the tensor-core path, with the fast
// exponential and division intrinsics: their few-ulp errors are far below
// the bf16 rounding of h that follows (relative 2^-9), and the epilogue is on
// the gate/up kernel's critical path (its single accumulator buffer waits
// for it).  For g below about -87 the divisor exceeds 2^126 (or is +inf)
// and __fdividef gives 0, silu's limit.
__device__ __forceinline__ float swiglu_fast(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Active experts in id order (warp-wide); buckets cut into chunks of kBN pairs.
// Buckets clamped into [0, P] (offsets that are not a valid bucketing give
// wrong sums, never an out-of-range pair).
// s_act holds weight-array indices (arena slots when expert_slot is given;
// experts without a slot are left out).
__device__ void tc_build_active(const int32_t* offsets, int E, int P, int* s_act, int* s_beg, int* s_end, int* s_cb,
                                int* s_n, const int32_t* expert_slot, int n_slots) {
    const int lane = threadIdx.x & 31;
    int lo[MOE_MAX_EXPERTS / 32], hi[MOE_MAX_EXPERTS / 32], wi[MOE_MAX_EXPERTS / 32];
#pragma unroll
    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) {
        const int e = 32 * j + lane;
        const int a = e < E ? __ldcg(offsets + e) : 0;
        const int b = e < E ? __ldcg(offsets + e + 1) : 0;
        wi[j] = e < E ? weight_index(expert_slot, n_slots, e) : -1;
        lo[j] = min(max(a, 0), P);
        hi[j] = wi[j] < 0 ? lo[j] : min(max(b, lo[j]), P);
    }
    int n = 0, nc = 0;
#pragma unroll
    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) {
        const bool a = hi[j] > lo[j];
        const uint32_t m = __ballot_sync(0xffffffffu, a);
        const int my_c = a ? (hi[j] - lo[j] + kBN - 1) / kBN : 0;
        int incl = my_c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (a) {
            const int jj = n + __popc(m & ((1u << lane) - 1u));
            s_act[jj] = wi[j];
            s_beg[jj] = lo[j];
            s_end[jj] = hi[j];
            s_cb[jj] = nc + incl - my_c;
        }
        n += __popc(m);
        nc += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
        *s_n = n;
        s_cb[n] = nc;
    }
}

struct Unit {
    int e, m0, p0, nv, N;  // expert, first weight row, first pair, valid pairs, MMA N
};

// Unit u -> (expert, weight-row tile, token chunk).  band = 0: chunk-major
// (a chunk's row tiles back to back, so its activations are reused at once).
// band > 0 (the reuse-ordering traversal of
// expxa.com/research/reuse-ordering-qualification, "What changed from the
// first experiment"): within each expert, row tiles go in bands of `band`,
// and a band visits every token chunk of the expert before the next band,
// so each weight tile is reused across the expert's chunks sooner.  Each
// expert keeps its own range of units, so both orders are a permutation of
// the same units and every unit's arithmetic is unchanged.
__device__ __forceinline__ Unit decode_unit(int u, int mt, const int* s_act, const int* s_beg, const int* s_end,
                                            const int* s_cb, int n, int band) {
    int g = u / mt;
    int m = u - g * mt;
    Unit U;
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_cb[mid] <= g) lo = mid;
        else hi = mid - 1;
    }
    if (band > 0) {
        const int nch = s_cb[lo + 1] - s_cb[lo];
        const int v = u - s_cb[lo] * mt;  // unit within the expert
        const int b = v / (band * nch), r = v - b * (band * nch);
        g = s_cb[lo] + r / band;
        m = b * band + r % band;
    }
    U.m0 = m * kBM;
    U.e = s_act[lo];
    U.p0 = s_beg[lo] + (g - s_cb[lo]) * kBN;
    U.nv = min(kBN, s_end[lo] - U.p0);
    U.N = (U.nv + 15) & ~15;
    return U;
}

__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, int32_t* status, volatile int* abort_flag) {
    if (mbar_wait(bar, parity)) return true;
    flag_status(status, MOE_STATUS_TIMEOUT_BIT);
    *abort_flag = 1;
    return false;
}

template <int NMAT, int EPI, int FMT>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_ffn_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                  const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_s0,
                  const __grid_constant__ CUtensorMap tm_s1, TcParams p) {
    constexpr int kRS = TcRing<NMAT>::RS;
    constexpr int AS = TcRing<NMAT>::AS;
    constexpr int NBUF = TcRing<NMAT>::NBUF;
    constexpr uint32_t kTmemCols = 512;  // accumulators, then the A operand stages
    constexpr uint32_t kAcol0 = TcRing<NMAT>::ACC_COLS;
    constexpr int kKR = FMT ? 2 * kBKR : kBKR;  // K per raw stage: 128 bytes of every row
    constexpr int kOps = kKR / kBK;             // operand stages per raw stage (2 or 4)
    extern __shared__ unsigned char tc_smem_raw[];
    __shared__ __align__(8) uint64_t raw_full[kRS], raw_empty[kRS], b_full[AS], a_full[AS], ab_empty[AS];
    __shared__ __align__(8) uint64_t acc_full[NBUF], acc_empty[NBUF], drain_bar;
    __shared__ int s_act[MOE_MAX_EXPERTS], s_beg[MOE_MAX_EXPERTS], s_end[MOE_MAX_EXPERTS];
    __shared__ int s_cb[MOE_MAX_EXPERTS + 1], s_n;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ int s_ep_tok[kBN];
    __shared__ float s_ep_w[kBN];

    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* raw = smem;                                   // [kRS][NMAT][kTile]
    unsigned char* Bs = raw + kRS * NMAT * kTile;                // [AS][kTile]
    unsigned char* Ss = Bs + AS * kTile;                         // [kRS][NMAT][128 rows][8 scales]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRS; ++s) {
            mbar_init(raw_full + s, 1);
            mbar_init(raw_empty + s, kDqWarps);
        }
        for (int s = 0; s < AS; ++s) {
            mbar_init(b_full + s, 1);
            mbar_init(a_full + s, kDqWarps);
            mbar_init(ab_empty + s, 1);
        }
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_empty + b, kEpWarps);
        }
        mbar_init(&drain_bar, 1);
        s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&s_tmem, kTmemCols);
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_a0);
        prefetch_tmap(&tm_s0);
        if (NMAT == 2) {
            prefetch_tmap(&tm_a1);
            prefetch_tmap(&tm_s1);
        }
        prefetch_tmap(&tm_b);
    }
    // Only the token producer waits for the previous kernel in the stream:
    // it alone reads what that kernel wrote (the gathered bf16 x, or h).
    // The weights, the bucketing, the routing weights and the arena's slots
    // were complete before that kernel let this grid launch (it waits for
    // its own predecessor first), so the active experts, the weight stream
    // and its dequantisation start at once, overlapping the previous
    // kernel's tail.  The combine target out is touched only by the down
    // projection's epilogue, after MMAs that follow the token producer's
    // wait (by then every kernel before this one has completed).
    if (warp == 2) tc_build_active(p.offsets, p.E, p.T * p.k, s_act, s_beg, s_end, s_cb, &s_n, p.eslot, p.nslots);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_launch_dependents();
    const uint32_t tmem = s_tmem;
    const int mt = p.rows / kBM;
    const int n_units = s_cb[s_n] * mt;
    const int kr_n = p.K / kKR;

    if (warp == 0) {
        // ------------------------------------------------- TMA producer: weights
        // runs ahead of the dequant warps by up to kRS raw stages, independent
        // of the operand ring (token tiles have their own producer, warp 2)
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            uint32_t rc = 0;
            for (int u = blockIdx.x; u < n_units && !s_abort; u += gridDim.x) {
                const Unit U = decode_unit(u, mt, s_act, s_beg, s_end, s_cb, s_n, p.band);
                const int wrow = U.e * p.rows + U.m0;
                for (int kr = 0; kr < kr_n; ++kr) {
                    const int rs = rc % kRS;
                    if (!tc_wait(raw_empty + rs, ((rc / kRS) & 1) ^ 1, p.status, &s_abort)) break;
                    mbar_arrive_expect_tx(raw_full + rs, NMAT * (kTile + kScTile));
                    // the stage's 128 bytes of every weight row (Q8_0: 128 K in four
                    // blocks; Q4_0: 256 K in eight), and a 16-byte aligned window
                    // of eight fp16 scales per row that holds those blocks
                    const int sx = FMT ? 8 * kr : (4 * kr) & ~7;
                    tma_load_2d_hint(raw + (rs * NMAT + 0) * kTile, &tm_a0, kr * kBKR, wrow, raw_full + rs, pol);
                    tma_load_2d(Ss + (rs * NMAT + 0) * kScTile, &tm_s0, sx, wrow, raw_full + rs);
                    if (NMAT == 2) {
                        tma_load_2d_hint(raw + (rs * NMAT + 1) * kTile, &tm_a1, kr * kBKR, wrow, raw_full + rs, pol);
                        tma_load_2d(Ss + (rs * NMAT + 1) * kScTile, &tm_s1, sx, wrow, raw_full + rs);
                    }
                    ++rc;
                }
            }
            // drain: every issued copy has landed before the CTA can exit
            for (uint32_t c = (rc > kRS ? rc - kRS : 0); c < rc; ++c) mbar_wait(raw_full + c % kRS, (c / kRS) & 1);
        }
    } else if (warp == 2) {
        // ------------------------------------------------- TMA producer: tokens
        if (lane == 0) {
            pdl_wait();  // the previous kernel's activations are complete and visible
            uint32_t ac = 0;
            for (int u = blockIdx.x; u < n_units && !s_abort; u += gridDim.x) {
                const Unit U = decode_unit(u, mt, s_act, s_beg, s_end, s_cb, s_n, p.band);
                const int nb = (U.N + kBRows - 1) / kBRows;
                for (int ks = 0; ks < p.K / kBK && !s_abort; ++ks) {
                    const int s = ac % AS;
                    if (!tc_wait(ab_empty + s, ((ac / AS) & 1) ^ 1, p.status, &s_abort)) break;
                    mbar_arrive_expect_tx(b_full + s, nb * kBRows * 128);
                    for (int bb = 0; bb < nb; ++bb)
                        tma_load_2d(Bs + s * kTile + bb * kBRows * 128, &tm_b, ks * kBK, U.p0 + bb * kBRows,
                                    b_full + s);
                    ++ac;
                }
            }
            for (uint32_t c = (ac > AS ? ac - AS : 0); c < ac; ++c) mbar_wait(b_full + c % AS, (c / AS) & 1);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t ac = 0, uc = 0;
            for (int u = blockIdx.x; u < n_units && !s_abort; u += gridDim.x, ++uc) {
                const Unit U = decode_unit(u, mt, s_act, s_beg, s_end, s_cb, s_n, p.band);
                const int buf = uc % NBUF;
                if (!tc_wait(acc_empty + buf, ((uc / NBUF) & 1) ^ 1, p.status, &s_abort)) break;
                tc_fence_after();
                const uint32_t idesc = umma_idesc_bf16(kBM, U.N);
                const uint32_t dcol = tmem + buf * NMAT * kBN;
                for (int ks = 0; ks < p.K / kBK; ++ks) {
                    const int s = ac % AS;
                    if (!tc_wait(a_full + s, (ac / AS) & 1, p.status, &s_abort)) break;
                    if (!tc_wait(b_full + s, (ac / AS) & 1, p.status, &s_abort)) break;
                    tc_fence_after();
                    const uint64_t bdesc = umma_desc_sw128(Bs + s * kTile);
#pragma unroll
                    for (int mat = 0; mat < NMAT; ++mat) {
                        // A: 128 TMEM lanes (weight rows) x 64 bf16 (32 columns); 16 K = 8 columns per MMA
                        const uint32_t acol = tmem + kAcol0 + (uint32_t)(s * NMAT + mat) * TcRing<NMAT>::A_COLS;
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)  // B: 16 bf16 = 32 bytes = 2 descriptor units
                            umma_bf16_ta(dcol + mat * kBN, acol + 8 * kk, bdesc + 2 * kk, idesc, (ks | kk) != 0);
                    }
                    umma_commit(ab_empty + s);
                    ++ac;
                }
                if (s_abort) break;
                umma_commit(acc_full + buf);
            }
            // all MMAs issued by this thread complete before TMEM is released
            umma_commit(&drain_bar);
            mbar_wait(&drain_bar, 0);
        }
    } else if (warp >= kDqWarp0 && warp < kDqWarp0 + kDqWarps) {
        // ---------------------------------------------------------------- dequantisation
        // thread = (row r, part pq of the 64-K operand stage: kCpt 16-K chunks);
        // warp w holds rows of TMEM lane quadrant w % 4
        const int tq = (warp - kDqWarp0) * 32 + lane;
        const int r = tq & (kBM - 1), pq = tq >> 7;
        uint32_t rc = 0, ac = 0;
        for (int u = blockIdx.x; u < n_units && !s_abort; u += gridDim.x) {
            bool ok = true;
            for (int kr = 0; kr < kr_n && ok; ++kr) {
                const int rs = rc % kRS;
                if (!tc_wait(raw_full + rs, (rc / kRS) & 1, p.status, &s_abort)) {
                    ok = false;
                    break;
                }
                // the raw stage's operand stages two at a time: all their TMEM
                // stores in flight before one wait
                for (int jp = 0; jp < kOps / 2 && ok; ++jp) {
                    const int s0 = ac % AS, s1 = (ac + 1) % AS;
                    if (!tc_wait(ab_empty + s0, ((ac / AS) & 1) ^ 1, p.status, &s_abort) ||
                        !tc_wait(ab_empty + s1, (((ac + 1) / AS) & 1) ^ 1, p.status, &s_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int s = j ? s1 : s0;
                        const int js = 2 * jp + j;  // operand stage within the raw stage: 64 K, two blocks
#pragma unroll
                        for (int mat = 0; mat < NMAT; ++mat) {
                            const unsigned char* rt = raw + (rs * NMAT + mat) * kTile;
                            const __half* sc = reinterpret_cast<const __half*>(Ss + (rs * NMAT + mat) * kScTile);
                            // this thread's block of the stage, from the stage's scale window
                            const float d =
                                __half2float(sc[r * 8 + (FMT ? 0 : (4 * kr) & 7) + 2 * js + (pq * kCpt) / 2]);
                            const f32x2 dd = f2_pack(d, d);
                            const float c = (FMT ? -32776.0f : -32896.0f) * d;  // -(2^15 + 8 or 128) * d
                            const f32x2 cc = f2_pack(c, c);
                            uint32_t v[8 * kCpt];  // this thread's row: 16 * kCpt bf16 of the 64-K stage
                            if (FMT == 0) {
#pragma unroll
                                for (int i = 0; i < kCpt; ++i) {
                                    const uint4 q =
                                        *reinterpret_cast<const uint4*>(rt + sw128(r, 4 * js + pq * kCpt + i));
                                    uint4 o0, o1;
                                    dequant16(q, dd, cc, o0, o1);
                                    v[8 * i + 0] = o0.x, v[8 * i + 1] = o0.y, v[8 * i + 2] = o0.z;
                                    v[8 * i + 3] = o0.w, v[8 * i + 4] = o1.x, v[8 * i + 5] = o1.y;
                                    v[8 * i + 6] = o1.z, v[8 * i + 7] = o1.w;
                                }
                            } else {  // one 16-byte chunk = one whole block of 32 values
                                dequant32_q4(*reinterpret_cast<const uint4*>(rt + sw128(r, 2 * js + pq)), dd, cc, v);
                            }
                            // TMEM lane = weight row (this warp's lane quadrant), 8 columns = 16 bf16 per chunk
                            tmem_st<8 * kCpt>(tmem + ((uint32_t)(r & ~31) << 16) + kAcol0 +
                                                  (uint32_t)(s * NMAT + mat) * TcRing<NMAT>::A_COLS + 8 * kCpt * pq,
                                              v);
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(a_full + s0);
                        mbar_arrive(a_full + s1);
                    }
                    ac += 2;
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(raw_empty + rs);
                ++rc;
                ok = !s_abort;
            }
            if (!ok) break;
        }
    } else if (warp >= kEpWarp0) {
        // ---------------------------------------------------------------- epilogue
        // kEpWarps warps: warp % 4 picks the TMEM lane quadrant (weight rows),
        // ep_half = which 16-column chunks (tokens) of the accumulator
        const int ew = warp % 4;
        const int ep_half = (warp - kEpWarp0) / 4;
        const int row = ew * 32 + lane;                 // weight row within the unit
        const int et = (warp - kEpWarp0) * 32 + lane;  // pair slot staged by this thread (if < kBN)
        constexpr int kEpThreads = kEpWarps * 32;
        uint32_t uc = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++uc) {
            // the epilogue warps leave together or not at all: they meet at
            // named barrier 2 below, so one warp leaving alone would strand
            // the others there
            if (!named_bar_and(2, kEpThreads, !s_abort)) break;
            const Unit U = decode_unit(u, mt, s_act, s_beg, s_end, s_cb, s_n, p.band);
            if (EPI == 1) {
                if (et < kBN) {
                    int tok = -1;
                    float w = 0.f;
                    if (et < U.nv) {
                        const int pp = U.p0 + et;
                        const int t = __ldcg(p.pair_tok + pp), sl = __ldcg(p.pair_slot + pp);
                        if (t >= 0 && t < p.T && sl >= 0 && sl < p.k) {
                            tok = t;
                            w = __ldcg(p.wts + (size_t)t * p.k + sl);
                        }
                    }
                    s_ep_tok[et] = tok;
                    s_ep_w[et] = w;
                }
                named_bar(2, kEpThreads);
            }
            const int buf = uc % NBUF;
            const bool landed = tc_wait(acc_full + buf, (uc / NBUF) & 1, p.status, &s_abort);
            if (!named_bar_and(2, kEpThreads, landed)) break;  // a timeout in any epilogue warp ends them all
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(ew * 32) << 16) + buf * NMAT * kBN;
            for (int c0 = 16 * ep_half; c0 < U.N; c0 += 16 * (kEpWarps / 4)) {
                float g[16], v[16];
                tmem_ld16(tbase + c0, g);
                if (NMAT == 2) tmem_ld16(tbase + kBN + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int n = c0 + i;
                    if (n < U.nv) {
                        const size_t pp = (size_t)(U.p0 + n);
                        if (EPI == 0) {
                            p.h[pp * p.rows + U.m0 + row] = __float2bfloat16_rn(swiglu_fast(g[i], v[i]));
                        } else if (EPI == 1) {
                            const int tok = s_ep_tok[n];
                            if (tok >= 0) atomicAdd(p.out + (size_t)tok * p.rows + U.m0 + row, s_ep_w[n] * g[i]);
                        } else {
                            p.out[pp * p.rows + U.m0 + row] = g[i];
                        }
                    }
                }
            }
            tc_fence_before();
            named_bar(2, kEpThreads);  // every epilogue thread is done with this buffer and the staged pairs
            if (lane == 0) mbar_arrive(acc_empty + buf);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// x (fp32, token order) -> xb (bf16, bucket order); also the combine target
// out = residual ? x : 0 for the down kernel's atomics.
__global__ void gather_bf16_kernel(const float* __restrict__ x, int T, int dm, const int32_t* __restrict__ pair_tok,
                                   const int32_t* __restrict__ offsets, int E, int P, __nv_bfloat16* __restrict__ xb,
                                   float* __restrict__ out_init, int residual, int init_early) {
    // The combine target first when the preceding kernel is this library's
    // routing, bucketing or arena admission of the same call: none of them
    // writes x or reads or writes out (out never aliases x), and every
    // kernel before them was complete before they let this grid launch, so
    // out is initialised while they still run.
    if (out_init && init_early) {
        const size_t n4 = (size_t)T * dm / 4;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
            reinterpret_cast<float4*>(out_init)[i] =
                residual ? __ldcg(reinterpret_cast<const float4*>(x) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_wait();  // the bucketing (pair_tok, offsets) is complete
    pdl_launch_dependents();
    if (out_init && !init_early) {
        const size_t n4 = (size_t)T * dm / 4;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
            reinterpret_cast<float4*>(out_init)[i] =
                residual ? __ldcg(reinterpret_cast<const float4*>(x) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int pv = __ldcg(offsets + E);
    const int c8 = dm / 8;  // 16-byte output chunks per row
    // one warp per pair row: lane c converts 8 values (two float4 of x) into
    // one 16-byte chunk, consecutive lanes on consecutive chunks
    const int lane = threadIdx.x & 31;
    const int nw = (int)(gridDim.x * blockDim.x) >> 5;
    for (int pp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); pp < P; pp += nw) {
        const int t = pp < pv ? __ldcg(pair_tok + pp) : -1;
        uint4* dst = reinterpret_cast<uint4*>(xb) + (size_t)pp * c8;
        if (t >= 0 && t < T) {
            const float4* src = reinterpret_cast<const float4*>(x + (size_t)t * dm);
            for (int c = lane; c < c8; c += 32) {
                const float4 a = __ldcg(src + 2 * c), b = __ldcg(src + 2 * c + 1);
                dst[c] = make_uint4(bf16x2_rn(a.x, a.y), bf16x2_rn(a.z, a.w), bf16x2_rn(b.x, b.y),
                                    bf16x2_rn(b.z, b.w));
            }
        } else {
            for (int c = lane; c < c8; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
        }
    }
}

// ------------------------------------------------------------------ host side
// Looked up once (racing first calls store the same pointer).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 f0 = fn.load(std::memory_order_acquire);
    if (!f0) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f0 = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
            fn.store(f0, std::memory_order_release);
        }
        cudaGetLastError();
    }
    return f0;
}

// 2-D K-major map: inner dimension K (elements), outer `rows`, box {bx, by},
// 128-byte swizzle (or none).
bool make_tmap(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t K, uint64_t rows,
               uint32_t bx, uint32_t by, bool swizzle = true) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K * (uint64_t)esize};
    const cuuint32_t box[2] = {bx, by};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_num_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

template <int NMAT, int EPI, int FMT>
cudaError_t launch_tc(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b, const CUtensorMap& s0,
                      const CUtensorMap& s1, const TcParams& p, cudaStream_t s) {
    constexpr int kRS = TcRing<NMAT>::RS;
    constexpr int AS = TcRing<NMAT>::AS;
    const size_t smem = (size_t)(kRS * NMAT + AS) * kTile + (size_t)kRS * NMAT * kScTile + 1024;
    auto kern = tc_ffn_kernel<NMAT, EPI, FMT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tc_num_sms(), 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a0, a1, b, s0, s1, p);
}

}  // namespace

bool ffn_tc_supported(const moe_layer_w& w, int T) {
    // K a multiple of 256: whole raw stages (128 K of Q8_0, 256 K of Q4_0),
    // and rows of scales (K / 32 fp16) a multiple of 16 bytes, as a tensor
    // map's row pitch must be
    return (w.wfmt == MOE_WFMT_Q8_0 || w.wfmt == MOE_WFMT_Q4_0) && w.d_model % 256 == 0 && w.d_ff % 256 == 0 && w.d_model % kBM == 0 &&
           w.d_ff % kBM == 0 && (long long)T * w.k >= kBN && encode_fn() != nullptr;
}

cudaError_t launch_ffn_tc(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                          const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse_combine,
                          float* out_or_ypairs, int residual, __nv_bfloat16* xb, __nv_bfloat16* hb, int32_t* status,
                          int reuse_order, int in_layer, cudaStream_t s) {
    const int P = T * w.k;
    const int dm = w.d_model, f = w.d_ff;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(tc_num_sms() * 4, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t err = cudaLaunchKernelEx(&cfg, gather_bf16_kernel, x, T, dm, pair_tok, offsets, w.E, P, xb,
                                             fuse_combine ? out_or_ypairs : (float*)nullptr, residual, in_layer);
        if (err != cudaSuccess) return err;
    }
    CUtensorMap tg, tu, td, txb, th, sg, su, sd;
    const uint64_t ns = (uint64_t)weight_slots(w);
    const int q4 = w.wfmt == MOE_WFMT_Q4_0;
    const uint64_t rb_gu = q4 ? dm / 2 : dm, rb_dn = q4 ? f / 2 : f;  // bytes per weight row
    if (!make_tmap(&tg, w.gate.qs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rb_gu, ns * f, kBKR, kBM) ||
        !make_tmap(&tu, w.up.qs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rb_gu, ns * f, kBKR, kBM) ||
        !make_tmap(&td, w.down.qs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rb_dn, ns * dm, kBKR, kBM) ||
        !make_tmap(&sg, w.gate.d, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, dm / 32, ns * f, 8, kBM, false) ||
        !make_tmap(&su, w.up.d, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, dm / 32, ns * f, 8, kBM, false) ||
        !make_tmap(&sd, w.down.d, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, f / 32, ns * dm, 8, kBM, false) ||
        !make_tmap(&txb, xb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dm, P, kBK, kBRows) ||
        !make_tmap(&th, hb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, f, P, kBK, kBRows))
        return cudaErrorInvalidValue;
    TcParams pg = {};
    pg.K = dm;
    pg.rows = f;
    pg.E = w.E;
    pg.T = T;
    pg.k = w.k;
    pg.offsets = offsets;
    pg.pair_tok = pair_tok;
    pg.pair_slot = pair_slot;
    pg.wts = wts;
    pg.d0 = w.gate.d;
    pg.d1 = w.up.d;
    pg.h = hb;
    pg.status = status;
    pg.eslot = w.expert_slot;
    pg.nslots = (int)ns;
    cudaError_t err = q4 ? launch_tc<2, 0, 1>(tg, tu, txb, sg, su, pg, s) : launch_tc<2, 0, 0>(tg, tu, txb, sg, su, pg, s);
    if (err != cudaSuccess) return err;
    TcParams pd = pg;
    pd.K = f;
    pd.rows = dm;
    pd.d0 = w.down.d;
    pd.d1 = nullptr;
    pd.h = nullptr;
    pd.out = out_or_ypairs;
    pd.band = (reuse_order && (dm / kBM) % kReuseBand == 0) ? kReuseBand : 0;
    if (q4) {
        if (fuse_combine) return launch_tc<1, 1, 1>(td, td, th, sd, sd, pd, s);
        return launch_tc<1, 2, 1>(td, td, th, sd, sd, pd, s);
    }
    if (fuse_combine) return launch_tc<1, 1, 0>(td, td, th, sd, sd, pd, s);
    return launch_tc<1, 2, 0>(td, td, th, sd, sd, pd, s);
}

}  // namespace moe
