// Shared device helpers and kernel-launcher declarations of libmoe_gb300.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kWarp = 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum over aligned groups of G lanes (G a power of two <= 32); every lane of a
// group ends with the same value (xor butterfly: each step adds the same two
// operands in both partner lanes).
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// 16-byte streaming load of weights: read once per kernel, so skip L1.
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float ldg_half(const uint16_t* p) {
    unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __half2float(__ushort_as_half(b));
}

// Four Q8_0 values in a 32-bit word of the device layout (bytes u = q + 128)
// -> four exact fp32 values q: each byte goes into the low mantissa byte of
// 2^23 (0x4B0000uu = 8388608 + u) and 8388608 + 128 is subtracted; every
// step is exact.
__device__ __forceinline__ float4 i8x4_to_f32x4(uint32_t w) {
    const uint32_t u = w;
    float4 r;
    r.x = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)) - 8388736.0f;
    r.y = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541)) - 8388736.0f;
    r.z = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)) - 8388736.0f;
    r.w = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543)) - 8388736.0f;
    return r;
}

__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
    acc = fmaf(a.x, b.x, acc);
    acc = fmaf(a.y, b.y, acc);
    acc = fmaf(a.z, b.z, acc);
    acc = fmaf(a.w, b.w, acc);
    return acc;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ void flag_status(int32_t* status, int bits) {
    if (status) atomicOr(status, bits);
}

// Index of expert e's matrices along the expert dimension of the weight
// arrays: e itself, or its arena slot (-1 when it has none in [0, n_slots)).
__device__ __forceinline__ int weight_index(const int32_t* expert_slot, int n_slots, int e) {
    if (!expert_slot) return e;
    const int s = __ldcg(expert_slot + e);
    return (s >= 0 && s < n_slots) ? s : -1;
}

// Entries of the weight arrays along the expert dimension.
inline int weight_slots(const moe_layer_w& w) { return w.expert_slot ? w.n_slots : w.E; }

// ---- launchers (defined in the kernel .cu files) --------------------------
// Router (+ the bucketing too when every token fits one cluster tile and
// `bucketed` is non-null; *bucketed then tells whether it was done).
cudaError_t launch_route(const float* x, int T, const moe_layer_w& w, int32_t* idx, float* wts, int32_t* offsets,
                         int32_t* pair_tok, int32_t* pair_slot, int32_t* pos, bool* bucketed, cudaStream_t s);

cudaError_t launch_bucket(const int32_t* idx, int T, int k, int E, int32_t* offsets, int32_t* pair_tok,
                          int32_t* pair_slot, int32_t* pos, int32_t* status, cudaStream_t s);

// fp32 expert path.  h: fp32 [P][d_ff] scratch.
cudaError_t launch_ffn_f32(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                           const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse_combine,
                           float* out_or_ypairs, int residual, float* h, cudaStream_t s);

// Streaming (persistent, bulk-copy pipelined) fp32 expert path for shapes
// with d_model, d_ff multiples of 64.
bool ffn_rows_supported(const moe_layer_w& w, int T);
cudaError_t launch_ffn_rows(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                            const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse_combine,
                            float* out_or_ypairs, int residual, float* h, cudaStream_t s);
bool ffn_stream_supported(const moe_layer_w& w);
bool ffn_stream_fits(const moe_layer_w& w, int T);  // shared memory of the configuration picked for T
cudaError_t launch_ffn_stream(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                              const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse_combine,
                              float* out_or_ypairs, int residual, float* h, int32_t* status, cudaStream_t s);

// Tensor-core (tcgen05) bf16 expert path for prefill-size batches.
// in_layer: the preceding kernel in the stream is this library's routing,
// bucketing or arena admission of the same layer call (none of them reads or
// writes out), so out may be initialised before that kernel completes.
bool ffn_tc_supported(const moe_layer_w& w, int T);
cudaError_t launch_ffn_tc(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                          const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse_combine,
                          float* out_or_ypairs, int residual, __nv_bfloat16* xb, __nv_bfloat16* hb, int32_t* status,
                          int reuse_order, int in_layer, cudaStream_t s);

// The whole layer for T <= 2 decode tokens in one cooperative launch (fp32
// path).  logits: [T][E] scratch; h: [T*k][d_ff] scratch; sync: 2 words.
bool decode_fused_supported(const moe_layer_w& w, int T);
cudaError_t launch_decode_fused(const float* x, int T, const moe_layer_w& w, int residual, float* out,
                                int32_t* idx_out, float* wts_out, int32_t* offsets_out, float* logits, float* h,
                                unsigned int* sync, int32_t* status, cudaStream_t s);

// The whole layer for T <= 2 decode tokens in one cooperative launch with a
// single grid-wide exchange (the router logits), the down projection split
// along K with each CTA's gate/up features (Q8_0, fp32 path).  lgw:
// decode_split_words(T, E) 8-byte workspace words, epoch: one 4-byte
// workspace word (any contents; calls sharing a workspace must not overlap).
bool decode_split_supported(const moe_layer_w& w, int T);
cudaError_t launch_decode_split(const float* x, int T, const moe_layer_w& w, int residual, float* out,
                                int32_t* idx_out, float* wts_out, int32_t* offsets_out, unsigned long long* lgw,
                                unsigned int* epoch, int32_t* status, cudaStream_t s);
size_t decode_split_words(int T, int E);

cudaError_t launch_pack_q8(const uint8_t* blocks, long long rows, int K, int8_t* qs, uint16_t* d, cudaStream_t s);
cudaError_t launch_pack_q4(const uint8_t* blocks, long long rows, int K, uint8_t* qs, uint16_t* d, cudaStream_t s);

cudaError_t launch_combine(const float* ypairs, const float* wts, const int32_t* pos, int T, int k, int dm,
                           const float* residual, float* out, cudaStream_t s);

// Expert arena (arena.cu).
size_t arena_blob_bytes(const moe_layer_w& w);
size_t arena_state_bytes(int L, int E, int S);
cudaError_t launch_arena_init(void* state, int L, int E, int S, cudaStream_t s);
cudaError_t launch_arena_pack_blob(const moe_layer_w& w, int layer, int e, void* blob, cudaStream_t s);
cudaError_t launch_arena_admit(void* state, int layer, const int32_t* offsets, int P, const void* host_blobs,
                               const moe_layer_w& arena, int32_t* slot_map, int32_t* status, cudaStream_t s);

}  // namespace moe
