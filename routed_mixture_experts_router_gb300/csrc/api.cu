// C ABI of libmoe_gb300: argument checks, workspace carving and the launch
// sequence of the routed MoE layer.  Every entry point only enqueues work on
// the caller's stream; nothing here synchronises or reads back.
#include <atomic>
#include <limits.h>

#include "common.cuh"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;

inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct WsLayout {
    size_t idx, wts, off, ptok, pslot, pos, h, xb, ypairs, lg, sync, smap, total;
};

// Workspace carve-up shared by every entry point: the routing results, the
// bucketing, the SwiGLU activations h [P][d_ff] and, for the deterministic
// combine, the per-pair outputs [P][d_model].
WsLayout ws_layout(int T, const moe_layer_w& w, int act, int flags) {
    const size_t P = (size_t)T * w.k;
    WsLayout L{};
    size_t o = 0;
    L.idx = o;    o = align_up(o + P * sizeof(int32_t));
    L.wts = o;    o = align_up(o + P * sizeof(float));
    L.off = o;    o = align_up(o + (size_t)(w.E + 1) * sizeof(int32_t));
    L.ptok = o;   o = align_up(o + P * sizeof(int32_t));
    L.pslot = o;  o = align_up(o + P * sizeof(int32_t));
    L.pos = o;    o = align_up(o + P * sizeof(int32_t));
    L.h = o;      o = align_up(o + P * (size_t)w.d_ff * sizeof(float));   // fp32 h, or bf16 h
    L.xb = o;                                                              // bf16 activations, bucket order
    if (act == MOE_ACT_BF16) o = align_up(o + P * (size_t)w.d_model * sizeof(uint16_t));
    L.ypairs = o;
    if (flags & MOE_FLAG_DETERMINISTIC) o = align_up(o + P * (size_t)w.d_model * sizeof(float));
    L.lg = o;                                                               // router logits (decode kernels)
    o = align_up(o + (T >= 1 && T <= 2 ? decode_split_words(T, w.E) : (size_t)T * w.E) * sizeof(unsigned long long));
    L.sync = o;   o = align_up(o + 2 * sizeof(unsigned int));               // grid-barrier words (fused decode)
    L.smap = o;   o = align_up(o + (size_t)w.E * sizeof(int32_t));           // expert -> arena slot map
    L.total = o;
    return L;
}

bool valid_geometry(const moe_layer_w* w) {
    if (!w) return false;
    if (w->E < 1 || w->E > MOE_MAX_EXPERTS) return false;
    if (w->k < 1 || w->k > MOE_MAX_TOPK || w->k > w->E) return false;
    if (w->d_model < 32 || w->d_model % 32 || w->d_model > 8192) return false;
    if (w->d_ff < 32 || w->d_ff % 32 || w->d_ff > 8192) return false;
    return w->wfmt == MOE_WFMT_Q8_0 || w->wfmt == MOE_WFMT_Q4_0;
}

// Whether launch_ffn has a kernel for this call: Q4_0 experts run on the
// lane-per-row kernels, or with bf16 activations on the tensor-core kernels;
// an arena slot map only on the kernels that resolve it (lane-per-row,
// streaming, tensor-core), not on the fallback.
bool ffn_supported(const moe_layer_w* w, int T, int act) {
    if (w->wfmt == MOE_WFMT_Q4_0)
        return (act == MOE_ACT_BF16 && ffn_tc_supported(*w, T)) || ffn_rows_supported(*w, T > 0 ? T : 1);
    if (!w->expert_slot) return true;
    return (act == MOE_ACT_BF16 && ffn_tc_supported(*w, T)) || ffn_rows_supported(*w, T) ||
           (ffn_stream_supported(*w) && ffn_stream_fits(*w, T > 0 ? T : 1));
}

bool valid_T(int T, const moe_layer_w* w) { return T >= 0 && T <= 65536 && (long long)T * w->k <= INT_MAX / 2; }

bool valid_arena(const moe_layer_w* arena) { return arena->n_slots >= 1 && arena->n_slots <= 65536; }

bool valid_router(const moe_layer_w* w) {
    return w->router_w && aligned16(w->router_w) && (!w->router_bias || aligned16(w->router_bias));
}

bool valid_experts(const moe_layer_w* w) {
    const moe_q8_mat* m[3] = {&w->gate, &w->up, &w->down};
    for (auto* q : m)
        if (!q->qs || !q->d || !aligned16(q->qs) || !aligned16(q->d)) return false;
    if (w->expert_slot && (w->n_slots < 1 || w->n_slots > 65536)) return false;
    return true;
}

// sm_103 (GB300) only: the library is built for sm_103a.
// The per-device answer is cached lock-free (threads racing on the first
// call store the same value).
int check_device() {
    static std::atomic<int> cached[64];  // 0 unknown, 1 ok, 2 unsupported (zero-initialised)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    int c = cached[dev].load(std::memory_order_relaxed);
    if (c == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        c = (major == 10 && minor == 3) ? 1 : 2;
        cached[dev].store(c, std::memory_order_relaxed);
    }
    return c == 1 ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

// Expert path: bf16 activations -> tcgen05 kernels when the batch fills at
// least one 128-pair MMA tile (smaller batches run the fp32 path, which is
// more accurate and memory-bound anyway); fp32 -> for 3+ tokens the
// lane-per-row kernels, for 1-2 tokens the streaming kernels, where the
// geometry allows; the per-expert-CTA kernels otherwise.  Q4_0 weights: the
// tensor-core kernels likewise, else the lane-per-row kernels for every T
// (the callers have checked the geometry).
cudaError_t launch_ffn(const float* x, int T, const moe_layer_w& w, int act, const int32_t* offsets,
                       const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse, float* out,
                       int residual, char* ws, const WsLayout& L, int32_t* status, cudaStream_t s,
                       int reuse_order = 0, int in_layer = 0) {
    float* h = reinterpret_cast<float*>(ws + L.h);
    if (act == MOE_ACT_BF16 && ffn_tc_supported(w, T))
        return launch_ffn_tc(x, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, residual,
                             reinterpret_cast<__nv_bfloat16*>(ws + L.xb), reinterpret_cast<__nv_bfloat16*>(h),
                             status, reuse_order, in_layer, s);
    if (w.wfmt != MOE_WFMT_Q8_0) {
        if (!ffn_rows_supported(w, T)) return cudaErrorNotSupported;
        return launch_ffn_rows(x, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, residual, h, s);
    }
    if (ffn_rows_supported(w, T))
        return launch_ffn_rows(x, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, residual, h, s);
    if (ffn_stream_supported(w) && ffn_stream_fits(w, T))
        return launch_ffn_stream(x, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, residual, h, status, s);
    if (w.expert_slot) return cudaErrorNotSupported;  // the per-expert-CTA kernels read weights in expert order
    return launch_ffn_f32(x, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, residual, h, s);
}

inline int cuda_rc(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    cudaGetLastError();
    return MOE_ERR_CUDA;
}

// An arena admission between the bucketing and the expert kernels.
struct ArenaCall {
    void* state;
    int layer;
    const void* host_blobs;
};

// Router (+ bucketing), optionally the arena admission, the expert FFNs and
// the combine.  idx, wts, off: where the routing and bucketing go.
cudaError_t layer_chain(const float* x, int T, const moe_layer_w& w, int act, int flags, int residual, float* out,
                        int32_t* idx, float* wts, int32_t* off, char* base, const WsLayout& L, int32_t* status,
                        const ArenaCall* arena, cudaStream_t s) {
    int32_t* ptok = reinterpret_cast<int32_t*>(base + L.ptok);
    int32_t* pslot = reinterpret_cast<int32_t*>(base + L.pslot);
    int32_t* pos = reinterpret_cast<int32_t*>(base + L.pos);
    bool bucketed = false;
    cudaError_t e = launch_route(x, T, w, idx, wts, off, ptok, pslot, pos, &bucketed, s);
    if (e != cudaSuccess) return e;
    if (!bucketed) {
        e = launch_bucket(idx, T, w.k, w.E, off, ptok, pslot, pos, status, s);
        if (e != cudaSuccess) return e;
    }
    moe_layer_w wf = w;
    if (arena) {
        int32_t* smap = reinterpret_cast<int32_t*>(base + L.smap);
        e = launch_arena_admit(arena->state, arena->layer, off, T * w.k, arena->host_blobs, w, smap, status, s);
        if (e != cudaSuccess) return e;
        wf.expert_slot = smap;
    }
    const int ro = (flags & MOE_FLAG_REUSE_ORDER) ? 1 : 0;
    if (flags & MOE_FLAG_DETERMINISTIC) {
        float* yp = reinterpret_cast<float*>(base + L.ypairs);
        e = launch_ffn(x, T, wf, act, off, ptok, pslot, wts, 0, yp, 0, base, L, status, s, ro, 1);
        if (e != cudaSuccess) return e;
        return launch_combine(yp, wts, pos, T, w.k, w.d_model, residual ? x : nullptr, out, s);
    }
    return launch_ffn(x, T, wf, act, off, ptok, pslot, wts, 1, out, residual, base, L, status, s, ro, 1);
}

}  // namespace

extern "C" {

const char* moe_version(void) { return "moe_gb300 0.1 (sm_103a)"; }

size_t moe_workspace_size(int T, const moe_layer_w* w, int act, int flags) {
    if (!valid_geometry(w) || !valid_T(T, w)) return 0;
    if (act != MOE_ACT_F32 && act != MOE_ACT_BF16) return 0;
    return ws_layout(T, *w, act, flags).total;
}

int moe_pack_q8(const uint8_t* blocks, long long rows, int K, int8_t* qs, uint16_t* d, void* stream) {
    if (rows < 0 || K <= 0 || K % 32) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!blocks || !qs || !d || !aligned16(qs)) return MOE_ERR_INVALID_ARG;
    int rc = check_device();
    if (rc) return rc;
    return cuda_rc(launch_pack_q8(blocks, rows, K, qs, d, (cudaStream_t)stream));
}

int moe_pack_q4(const uint8_t* blocks, long long rows, int K, uint8_t* qs, uint16_t* d, void* stream) {
    if (rows < 0 || K <= 0 || K % 32) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!blocks || !qs || !d || !aligned16(qs)) return MOE_ERR_INVALID_ARG;
    int rc = check_device();
    if (rc) return rc;
    return cuda_rc(launch_pack_q4(blocks, rows, K, qs, d, (cudaStream_t)stream));
}

int moe_route(const float* x, int T, const moe_layer_w* w, int32_t* idx, float* wts, void* stream) {
    if (!valid_geometry(w) || !valid_T(T, w)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !idx || !wts || !aligned16(x) || !valid_router(w)) return MOE_ERR_INVALID_ARG;
    int rc = check_device();
    if (rc) return rc;
    return cuda_rc(launch_route(x, T, *w, idx, wts, nullptr, nullptr, nullptr, nullptr, nullptr, (cudaStream_t)stream));
}

int moe_bucket(const int32_t* idx, int T, int k, int E, int32_t* offsets, int32_t* pair_tok, int32_t* pair_slot,
               int32_t* pos, int32_t* status, void* stream) {
    if (E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > MOE_MAX_TOPK || k > E || T < 0 || T > 65536)
        return MOE_ERR_INVALID_ARG;
    if (!offsets || (T > 0 && (!idx || !pair_tok || !pair_slot || !pos))) return MOE_ERR_INVALID_ARG;
    int rc = check_device();
    if (rc) return rc;
    return cuda_rc(launch_bucket(idx, T, k, E, offsets, pair_tok, pair_slot, pos, status, (cudaStream_t)stream));
}

int moe_expert_ffn_q8(const float* x, int T, const moe_layer_w* w, const int32_t* offsets, const int32_t* pair_tok,
                      const int32_t* pair_slot, const float* wts, int act, int fuse_combine, float* out_or_ypairs,
                      int residual, void* ws, size_t ws_bytes, int32_t* status, void* stream) {
    if (!valid_geometry(w) || !valid_T(T, w)) return MOE_ERR_INVALID_ARG;
    if (act != MOE_ACT_F32 && act != MOE_ACT_BF16) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !offsets || !pair_tok || !pair_slot || !wts || !out_or_ypairs || !aligned16(x) ||
        !aligned16(out_or_ypairs) || !valid_experts(w))
        return MOE_ERR_INVALID_ARG;
    if (fuse_combine && (const void*)out_or_ypairs == (const void*)x) return MOE_ERR_INVALID_ARG;
    if (!ffn_supported(w, T, act)) return MOE_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(T, *w, act, 0);
    if (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return MOE_ERR_WORKSPACE;
    int rc = check_device();
    if (rc) return rc;
    return cuda_rc(launch_ffn(x, T, *w, act, offsets, pair_tok, pair_slot, wts, fuse_combine ? 1 : 0, out_or_ypairs,
                              residual, static_cast<char*>(ws), L, status, (cudaStream_t)stream));
}

int moe_combine(const float* ypairs, const float* wts, const int32_t* pos, int T, int k, int d_model,
                const float* residual, float* out, void* stream) {
    if (T < 0 || k < 1 || k > MOE_MAX_TOPK || d_model < 32 || d_model % 32) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!ypairs || !wts || !pos || !out || !aligned16(ypairs) || !aligned16(out) ||
        (residual && !aligned16(residual)))
        return MOE_ERR_INVALID_ARG;
    int rc = check_device();
    if (rc) return rc;
    return cuda_rc(launch_combine(ypairs, wts, pos, T, k, d_model, residual, out, (cudaStream_t)stream));
}

int moe_layer_forward(const float* x, int T, const moe_layer_w* w, int act, int flags, int residual, float* out,
                      int32_t* idx_out, float* wts_out, int32_t* offsets_out, void* ws, size_t ws_bytes,
                      int32_t* status, void* stream) {
    if (!valid_geometry(w) || !valid_T(T, w)) return MOE_ERR_INVALID_ARG;
    if (act != MOE_ACT_F32 && act != MOE_ACT_BF16) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !out || !aligned16(x) || !aligned16(out) || (const void*)x == (const void*)out || !valid_router(w) ||
        !valid_experts(w))
        return MOE_ERR_INVALID_ARG;
    if (!ffn_supported(w, T, act)) return MOE_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(T, *w, act, flags);
    if (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return MOE_ERR_WORKSPACE;
    int rc = check_device();
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    char* base = static_cast<char*>(ws);
    int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(base + L.idx);
    float* wts = wts_out ? wts_out : reinterpret_cast<float*>(base + L.wts);
    int32_t* off = offsets_out ? offsets_out : reinterpret_cast<int32_t*>(base + L.off);
    // One or two decode tokens on the fp32 path: the whole layer in one
    // cooperative launch (falls through to the separate kernels if the device
    // cannot co-schedule it).
    const bool f32_path = act == MOE_ACT_F32 || !ffn_tc_supported(*w, T);
    if (f32_path && !(flags & MOE_FLAG_DETERMINISTIC) && decode_split_supported(*w, T)) {
        const cudaError_t fe = launch_decode_split(x, T, *w, residual, out, idx_out, wts_out, offsets_out,
                                                   reinterpret_cast<unsigned long long*>(base + L.lg),
                                                   reinterpret_cast<unsigned int*>(base + L.sync), status, s);
        if (fe == cudaSuccess) return MOE_OK;
        if (fe != cudaErrorInvalidConfiguration && fe != cudaErrorCooperativeLaunchTooLarge) return cuda_rc(fe);
        cudaGetLastError();
    }
    if (f32_path && !(flags & MOE_FLAG_DETERMINISTIC) && decode_fused_supported(*w, T)) {
        const cudaError_t fe = launch_decode_fused(x, T, *w, residual, out, idx_out, wts_out, offsets_out,
                                                   reinterpret_cast<float*>(base + L.lg),
                                                   reinterpret_cast<float*>(base + L.h),
                                                   reinterpret_cast<unsigned int*>(base + L.sync), status, s);
        if (fe == cudaSuccess) return MOE_OK;
        if (fe != cudaErrorCooperativeLaunchTooLarge && fe != cudaErrorInvalidConfiguration) return cuda_rc(fe);
        cudaGetLastError();
    }
    return cuda_rc(layer_chain(x, T, *w, act, flags, residual, out, idx, wts, off, base, L, status, nullptr, s));
}

size_t moe_arena_blob_bytes(const moe_layer_w* w) {
    if (!valid_geometry(w)) return 0;
    return arena_blob_bytes(*w);
}

size_t moe_arena_state_bytes(int layers, int experts, int slots) { return arena_state_bytes(layers, experts, slots); }

int moe_arena_init(void* state, int layers, int experts, int slots, void* stream) {
    if (!state || arena_state_bytes(layers, experts, slots) == 0 || (reinterpret_cast<uintptr_t>(state) & 255u))
        return MOE_ERR_INVALID_ARG;
    int rc = check_device();
    if (rc) return rc;
    return cuda_rc(launch_arena_init(state, layers, experts, slots, (cudaStream_t)stream));
}

int moe_arena_pack_blob(const moe_layer_w* w, int layer, int e, void* blob, void* stream) {
    if (!valid_geometry(w) || !valid_experts(w) || w->expert_slot) return MOE_ERR_INVALID_ARG;
    if (layer < 0 || e < 0 || e >= w->E || !blob || !aligned16(blob)) return MOE_ERR_INVALID_ARG;
    int rc = check_device();
    if (rc) return rc;
    return cuda_rc(launch_arena_pack_blob(*w, layer, e, blob, (cudaStream_t)stream));
}

int moe_arena_admit(void* state, int layer, const int32_t* offsets, int P, const void* host_blobs,
                    const moe_layer_w* arena, int32_t* slot_map, int32_t* status, void* stream) {
    if (!valid_geometry(arena) || !valid_arena(arena)) return MOE_ERR_INVALID_ARG;
    moe_layer_w a = *arena;
    a.expert_slot = nullptr;
    if (!valid_experts(&a) || !state || (reinterpret_cast<uintptr_t>(state) & 255u) || !offsets || P < 0 ||
        !host_blobs || !aligned16(host_blobs) || !slot_map || layer < 0)
        return MOE_ERR_INVALID_ARG;
    int rc = check_device();
    if (rc) return rc;
    return cuda_rc(launch_arena_admit(state, layer, offsets, P, host_blobs, a, slot_map, status, (cudaStream_t)stream));
}

int moe_layer_forward_arena(const float* x, int T, const moe_layer_w* w, int act, int flags, int residual,
                            float* out, void* state, int layer, const void* host_blobs, void* ws, size_t ws_bytes,
                            int32_t* status, void* stream) {
    if (!valid_geometry(w) || !valid_T(T, w) || !valid_arena(w)) return MOE_ERR_INVALID_ARG;
    if (act != MOE_ACT_F32 && act != MOE_ACT_BF16) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    moe_layer_w a = *w;
    a.expert_slot = nullptr;
    if (!x || !out || !aligned16(x) || !aligned16(out) || (const void*)x == (const void*)out || !valid_router(w) ||
        !valid_experts(&a) || !state || (reinterpret_cast<uintptr_t>(state) & 255u) || !host_blobs ||
        !aligned16(host_blobs) || layer < 0)
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, *w, act, flags);
    if (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return MOE_ERR_WORKSPACE;
    {
        moe_layer_w probe = a;
        probe.expert_slot = reinterpret_cast<const int32_t*>(static_cast<char*>(ws) + L.smap);
        if (!ffn_supported(&probe, T, act)) return MOE_ERR_UNSUPPORTED;
    }
    int rc = check_device();
    if (rc) return rc;
    char* base = static_cast<char*>(ws);
    const ArenaCall ac{state, layer, host_blobs};
    return cuda_rc(layer_chain(x, T, a, act, flags, residual, out, reinterpret_cast<int32_t*>(base + L.idx),
                               reinterpret_cast<float*>(base + L.wts), reinterpret_cast<int32_t*>(base + L.off), base,
                               L, status, &ac, (cudaStream_t)stream));
}

}  // extern "C"
