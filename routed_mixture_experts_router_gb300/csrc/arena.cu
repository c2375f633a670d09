// Expert arena: layer-qualified experts resident in HBM slots, with the miss
// path reading page-locked host memory directly.
//
// "Managed VRAM expert arena" and the miss path that "changes residency
// beneath the compute plane" (amalgafy.com/technical-overview, "VRAM budget
// policy", "Execution architecture"); blobs are page-aligned like the pages'
// expert blobs ("I/O path"; 5,017,600 B per Q8_0 expert of the qwen3_moe
// geometry, amalgafy.com/evidence, "Synthetic cache matrix").
//
// Everything runs on the GPU, in stream order, with no host readback: the
// admission kernel (one CTA) turns a layer's bucketing into hits, misses and
// LRU victims and updates the residency tables; the copy kernel (one CTA per
// SM pair) moves the missed blobs from host memory into their slots, reading
// the host memory over NVLink-C2C with ordinary 16-byte loads.  The FFN
// kernels then read the weights through the expert -> slot map.
//
// State layout (device memory, 256-byte aligned parts):
//   moe_arena_stats | slot_of int32 [L][E] | owner int32 [S] |
//   stamp uint32 [S] | miss_slot int32 [E] | miss_src int32 [E]
// slot_of[l*E+e] is e's slot in layer l (-1: not resident), owner[s] the key
// l*E+e held by slot s (-1: empty), stamp[s] the admission clock of its last
// use (0: never), miss_* the copies the latest admission asked for.
#include "common.cuh"

namespace moe {

namespace {

constexpr uint32_t kBlobMagic = 0x424f454du;  // bytes "MEOB" little endian
constexpr size_t kBlobHeader = 4096;
constexpr int kAdmitThreads = 1024;
constexpr int kMaxSlots = 65536;
constexpr int kNumSegs = 6;  // gate qs, up qs, down qs, gate d, up d, down d

__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct ArenaLayout {
    size_t slot_of, owner, stamp, miss_slot, miss_src, total;
};

__host__ __device__ inline ArenaLayout arena_layout(int L, int E, int S) {
    ArenaLayout A;
    size_t o = align256(sizeof(moe_arena_stats));
    A.slot_of = o;
    o = align256(o + (size_t)L * E * 4);
    A.owner = o;
    o = align256(o + (size_t)S * 4);
    A.stamp = o;
    o = align256(o + (size_t)S * 4);
    A.miss_slot = o;
    o = align256(o + (size_t)E * 4);
    A.miss_src = o;
    o = align256(o + (size_t)E * 4);
    A.total = o;
    return A;
}

// Byte sizes of the six payload segments of one expert, in payload order.
struct Segs {
    unsigned long long size[kNumSegs];
    unsigned char* base[kNumSegs];  // arena (or layer) arrays: segment i of slot s at base[i] + s * size[i]
};

Segs expert_segs(const moe_layer_w& w) {
    const bool q4 = w.wfmt == MOE_WFMT_Q4_0;
    const unsigned long long f = w.d_ff, dm = w.d_model;
    Segs g;
    g.size[0] = f * (q4 ? dm / 2 : dm);
    g.size[1] = g.size[0];
    g.size[2] = dm * (q4 ? f / 2 : f);
    g.size[3] = f * (dm / 32) * 2;
    g.size[4] = g.size[3];
    g.size[5] = dm * (f / 32) * 2;
    g.base[0] = (unsigned char*)w.gate.qs;
    g.base[1] = (unsigned char*)w.up.qs;
    g.base[2] = (unsigned char*)w.down.qs;
    g.base[3] = (unsigned char*)w.gate.d;
    g.base[4] = (unsigned char*)w.up.d;
    g.base[5] = (unsigned char*)w.down.d;
    return g;
}

unsigned long long payload_bytes(const Segs& g) {
    unsigned long long p = 0;
    for (int i = 0; i < kNumSegs; ++i) p += g.size[i];
    return p;
}

// ------------------------------------------------------------------- init --
__global__ void arena_init_kernel(unsigned char* state, int L, int E, int S) {
    const ArenaLayout A = arena_layout(L, E, S);
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x, nt = (size_t)gridDim.x * blockDim.x;
    if (tid == 0) {
        moe_arena_stats* st = reinterpret_cast<moe_arena_stats*>(state);
        st->hits = st->misses = st->bytes_in = 0ull;
        st->clock = 0u;
        st->layers = L;
        st->experts = E;
        st->slots = S;
        st->last_misses = 0;
        st->full_events = 0;
        st->reserved[0] = st->reserved[1] = 0;
    }
    int32_t* slot_of = reinterpret_cast<int32_t*>(state + A.slot_of);
    int32_t* owner = reinterpret_cast<int32_t*>(state + A.owner);
    uint32_t* stamp = reinterpret_cast<uint32_t*>(state + A.stamp);
    for (size_t i = tid; i < (size_t)L * E; i += nt) slot_of[i] = -1;
    for (size_t i = tid; i < (size_t)S; i += nt) {
        owner[i] = -1;
        stamp[i] = 0u;
    }
}

// ------------------------------------------------------------- blob pack --
__global__ void arena_pack_kernel(Segs g, int e, unsigned char* blob, uint32_t h0, uint32_t h1, uint32_t h2,
                                  uint32_t h3, uint32_t h4, uint32_t h5, uint32_t h6, uint32_t h7) {
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x, nt = (size_t)gridDim.x * blockDim.x;
    if (blockIdx.x == 0) {  // header page: 8 words, the rest zero
        uint32_t* hw = reinterpret_cast<uint32_t*>(blob);
        const uint32_t words[8] = {h0, h1, h2, h3, h4, h5, h6, h7};
        for (int i = threadIdx.x; i < (int)(kBlobHeader / 4); i += blockDim.x) hw[i] = i < 8 ? words[i] : 0u;
    }
    size_t off = kBlobHeader;
    for (int i = 0; i < kNumSegs; ++i) {
        const uint4* src = reinterpret_cast<const uint4*>(g.base[i] + (size_t)e * g.size[i]);
        uint4* dst = reinterpret_cast<uint4*>(blob + off);
        for (size_t q = tid; q < g.size[i] / 16; q += nt) dst[q] = src[q];
        off += g.size[i];
    }
    // tail padding to the page boundary
    const size_t end = (off + 4095) & ~(size_t)4095;
    for (size_t q = off / 16 + tid; q < end / 16; q += nt) reinterpret_cast<uint4*>(blob)[q] = make_uint4(0, 0, 0, 0);
}

// -------------------------------------------------------------- admission --
// Exclusive prefix over the block of one int per thread (kAdmitThreads
// threads); returns the thread's prefix, *total the block sum.
__device__ int block_excl_scan(int v, int* s_w, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kAdmitThreads / 32 ? s_w[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += t;
        }
        s_w[lane] = wi - w;  // exclusive per warp
        if (lane == 31) s_w[32] = wi;
    }
    __syncthreads();
    const int r = s_w[warp] + incl - v;
    *total = s_w[32];
    __syncthreads();  // s_w free for the next scan
    return r;
}

__global__ void __launch_bounds__(kAdmitThreads, 1)
    arena_admit_kernel(unsigned char* state, int layer, const int32_t* __restrict__ offsets, int P, int E, int S,
                       unsigned long long payload, int32_t* __restrict__ slot_map, int32_t* status) {
    __shared__ int s_act[MOE_MAX_EXPERTS], s_miss[MOE_MAX_EXPERTS], s_vic[MOE_MAX_EXPERTS];
    __shared__ uint32_t s_vstamp[MOE_MAX_EXPERTS];
    __shared__ int s_w[33];
    __shared__ unsigned int s_hist[256];
    __shared__ int s_ok, s_L, s_nact, s_nmiss, s_nvic, s_rank;
    __shared__ uint32_t s_clock, s_prefix, s_mask;
    moe_arena_stats* st = reinterpret_cast<moe_arena_stats*>(state);
    const int tid = threadIdx.x;
    if (tid == 0) {
        const int L = st->layers;
        s_ok = layer >= 0 && layer < L && st->experts == E && st->slots == S;
        s_L = L;
        if (s_ok) s_clock = ++st->clock;
    }
    __syncthreads();
    if (!s_ok) {  // the state was made for another geometry: map nothing
        for (int e = tid; e < E; e += kAdmitThreads) slot_map[e] = -1;
        if (tid == 0) flag_status(status, MOE_STATUS_BAD_INDEX);
        return;
    }
    const ArenaLayout A = arena_layout(s_L, E, S);
    int32_t* slot_of = reinterpret_cast<int32_t*>(state + A.slot_of);
    int32_t* owner = reinterpret_cast<int32_t*>(state + A.owner);
    uint32_t* stamp = reinterpret_cast<uint32_t*>(state + A.stamp);
    int32_t* miss_slot = reinterpret_cast<int32_t*>(state + A.miss_slot);
    int32_t* miss_src = reinterpret_cast<int32_t*>(state + A.miss_src);
    const uint32_t clock = s_clock;
    const int key0 = layer * E;

    // 1. active experts (non-empty clamped buckets), ascending
    int active = 0;
    if (tid < E) {
        const int lo = min(max(__ldcg(offsets + tid), 0), P);
        const int hi = min(max(__ldcg(offsets + tid + 1), lo), P);
        active = hi > lo;
    }
    int tot;
    const int ra = block_excl_scan(active, s_w, &tot);
    if (active) s_act[ra] = tid;
    if (tid == 0) s_nact = tot;
    __syncthreads();
    const int nact = s_nact;

    // 2. hits take this admission's stamp; misses listed ascending
    int miss = 0;
    if (tid < nact) {
        const int e = s_act[tid], key = key0 + e;
        const int s = slot_of[key];
        const bool hit = s >= 0 && s < S && owner[s] == key;
        if (hit) {
            stamp[s] = clock;
            slot_map[e] = s;
        }
        miss = !hit;
    }
    const int rm = block_excl_scan(miss, s_w, &tot);
    if (miss) s_miss[rm] = s_act[tid];
    if (tid == 0) s_nmiss = tot;
    __syncthreads();  // hit stamps and the miss list visible to the block
    const int nmiss = s_nmiss, nhit = nact - nmiss;
    const int need = min(nmiss, S - nhit);  // evictable slots: every slot but this admission's hits
    if (need > 0) {
        // 3. the need-th smallest stamp among evictable slots (stamp != clock),
        //    MSB-first radix select over the 32-bit stamps
        if (tid == 0) {
            s_prefix = 0u;
            s_mask = 0u;
            s_rank = need - 1;
        }
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += kAdmitThreads) s_hist[i] = 0u;
            __syncthreads();
            const uint32_t prefix = s_prefix, mask = s_mask;
            for (int s = tid; s < S; s += kAdmitThreads) {
                const uint32_t v = stamp[s];
                if (v != clock && (v & mask) == prefix) atomicAdd(&s_hist[(v >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (tid == 0) {
                int r = s_rank;
                uint32_t d = 0;
                for (; d < 256u; ++d) {
                    if ((int)s_hist[d] > r) break;
                    r -= (int)s_hist[d];
                }
                s_rank = r;  // rank among evictable slots with the chosen digits so far
                s_prefix = prefix | (d << shift);
                s_mask = mask | (255u << shift);
            }
            __syncthreads();
        }
        // 4. victims: every evictable slot with a smaller stamp, then the
        //    first rank+1 slots (ascending) with the threshold stamp
        const uint32_t vstar = s_prefix;
        const int take_eq = s_rank + 1;
        const int per = (S + kAdmitThreads - 1) / kAdmitThreads;  // contiguous slot range per thread
        const int s0 = min(tid * per, S), s1 = min(s0 + per, S);
        int neq = 0;
        for (int s = s0; s < s1; ++s) {
            const uint32_t v = stamp[s];
            neq += (v == vstar);  // vstar != clock, so these are evictable
        }
        int eq_before = block_excl_scan(neq, s_w, &tot);
        if (tid == 0) s_nvic = 0;
        __syncthreads();
        for (int s = s0; s < s1; ++s) {
            const uint32_t v = stamp[s];
            bool take = false;
            if (v != clock && v < vstar) take = true;
            if (v == vstar) take = eq_before++ < take_eq;
            if (take) {
                const int j = atomicAdd(&s_nvic, 1);
                if (j < MOE_MAX_EXPERTS) {
                    s_vic[j] = s;
                    s_vstamp[j] = v;
                }
            }
        }
        __syncthreads();
        // 5. victims in ascending (stamp, slot); miss j takes victim j
        int my_slot = -1, my_rank = 0;
        if (tid < need) {
            my_slot = s_vic[tid];
            const uint32_t my_v = s_vstamp[tid];
            for (int j = 0; j < need; ++j) {
                const uint32_t v = s_vstamp[j];
                my_rank += (v < my_v) || (v == my_v && s_vic[j] < my_slot);
            }
        }
        __syncthreads();
        if (tid < need) s_vic[my_rank] = my_slot;
        __syncthreads();
        if (tid < need) {
            const int e = s_miss[tid], key = key0 + e, s = s_vic[tid];
            const int old = owner[s];
            if (old >= 0 && old < s_L * E) slot_of[old] = -1;
            owner[s] = key;
            slot_of[key] = s;
            stamp[s] = clock;
            slot_map[e] = s;
            miss_slot[tid] = s;
            miss_src[tid] = key;
        }
    }
    for (int j = max(need, 0) + tid; j < nmiss; j += kAdmitThreads) slot_map[s_miss[j]] = -1;
    __syncthreads();  // this admission's evictions visible to the block
    // experts not routed this time: their slot after this admission, if any
    for (int e = tid; e < E; e += kAdmitThreads) {
        const int lo = min(max(__ldcg(offsets + e), 0), P);
        const int hi = min(max(__ldcg(offsets + e + 1), lo), P);
        if (hi <= lo) {
            const int s = slot_of[key0 + e];
            slot_map[e] = (s >= 0 && s < S && owner[s] == key0 + e) ? s : -1;
        }
    }
    if (tid == 0) {
        st->hits += (unsigned long long)nhit;
        st->misses += (unsigned long long)max(need, 0);
        st->bytes_in += (unsigned long long)max(need, 0) * payload;
        st->last_misses = max(need, 0);
        if (need < nmiss) {
            st->full_events += 1;
            flag_status(status, MOE_STATUS_ARENA_FULL);
        }
    }
}

// ------------------------------------------------------------------ copy --
// The blobs the latest admission asked for, host memory -> arena slots.
// Each blob's payload is read as one contiguous run of 16-byte pieces (all
// threads on it, 8 independent loads in flight per thread); piece q goes to
// the segment whose range holds it.
constexpr int kCopyUnroll = 8;

__device__ __forceinline__ uint4* copy_dst(const Segs& g, const unsigned long long (&c)[kNumSegs + 1], size_t slot,
                                           size_t q) {
    unsigned char* base = g.base[0];
    unsigned long long size = g.size[0], start = 0;
#pragma unroll
    for (int k = 1; k < kNumSegs; ++k) {  // constant indices only: the parameters stay in registers
        if (q >= c[k]) {
            base = g.base[k];
            size = g.size[k];
            start = c[k];
        }
    }
    return reinterpret_cast<uint4*>(base + slot * size) + (q - start);
}

__global__ void __launch_bounds__(256) arena_copy_kernel(const unsigned char* state, const unsigned char* host_blobs,
                                                         unsigned long long blob_bytes, Segs g) {
    const moe_arena_stats* st = reinterpret_cast<const moe_arena_stats*>(state);
    const int n = st->last_misses;
    if (n <= 0) return;
    const ArenaLayout A = arena_layout(st->layers, st->experts, st->slots);
    const int32_t* miss_slot = reinterpret_cast<const int32_t*>(state + A.miss_slot);
    const int32_t* miss_src = reinterpret_cast<const int32_t*>(state + A.miss_src);
    unsigned long long c[kNumSegs + 1];  // segment starts in 16-byte pieces
    c[0] = 0;
#pragma unroll
    for (int i = 0; i < kNumSegs; ++i) c[i + 1] = c[i] + g.size[i] / 16;
    const size_t p16 = c[kNumSegs];
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x, nt = (size_t)gridDim.x * blockDim.x;
    for (int j = 0; j < n; ++j) {
        const size_t slot = (size_t)miss_slot[j];
        const uint4* s4 = reinterpret_cast<const uint4*>(host_blobs + (size_t)miss_src[j] * blob_bytes + kBlobHeader);
        for (size_t q0 = tid; q0 < p16; q0 += kCopyUnroll * nt) {
            uint4 v[kCopyUnroll];
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) {
                const size_t q = q0 + u * nt;
                if (q < p16) v[u] = s4[q];
            }
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) {
                const size_t q = q0 + u * nt;
                if (q < p16) *copy_dst(g, c, slot, q) = v[u];
            }
        }
    }
}

int arena_num_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

}  // namespace

size_t arena_blob_bytes(const moe_layer_w& w) {
    const unsigned long long p = payload_bytes(expert_segs(w));
    return kBlobHeader + (size_t)((p + 4095) & ~4095ull);
}

size_t arena_state_bytes(int L, int E, int S) {
    if (L < 1 || E < 1 || E > MOE_MAX_EXPERTS || S < 1 || S > kMaxSlots) return 0;
    if ((long long)L * E > (1ll << 30)) return 0;
    return arena_layout(L, E, S).total;
}

cudaError_t launch_arena_init(void* state, int L, int E, int S, cudaStream_t s) {
    arena_init_kernel<<<arena_num_sms(), 256, 0, s>>>(static_cast<unsigned char*>(state), L, E, S);
    return cudaGetLastError();
}

cudaError_t launch_arena_pack_blob(const moe_layer_w& w, int layer, int e, void* blob, cudaStream_t s) {
    const Segs g = expert_segs(w);
    const unsigned long long p = payload_bytes(g);
    arena_pack_kernel<<<arena_num_sms(), 256, 0, s>>>(g, e, static_cast<unsigned char*>(blob), kBlobMagic, 1u,
                                                      (uint32_t)w.wfmt, (uint32_t)layer, (uint32_t)e,
                                                      (uint32_t)w.d_model, (uint32_t)w.d_ff, (uint32_t)p);
    return cudaGetLastError();
}

cudaError_t launch_arena_admit(void* state, int layer, const int32_t* offsets, int P, const void* host_blobs,
                               const moe_layer_w& arena, int32_t* slot_map, int32_t* status, cudaStream_t s) {
    const Segs g = expert_segs(arena);
    unsigned char* st = static_cast<unsigned char*>(state);
    arena_admit_kernel<<<1, kAdmitThreads, 0, s>>>(st, layer, offsets, P, arena.E, arena.n_slots, payload_bytes(g),
                                                   slot_map, status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    arena_copy_kernel<<<2 * arena_num_sms(), 256, 0, s>>>(st, static_cast<const unsigned char*>(host_blobs),
                                                          (unsigned long long)arena_blob_bytes(arena), g);
    return cudaGetLastError();
}

}  // namespace moe
