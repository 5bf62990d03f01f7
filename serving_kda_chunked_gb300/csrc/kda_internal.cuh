// kda_internal.cuh -- shared declarations of the KDA CUDA library (internal).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// Arguments of one prefill call after host validation.
struct PrefillArgs {
    const void *q, *k, *v;
    const float *g, *beta, *S0;
    const int32_t *cu_seqlens;
    void *o;
    float *S_T;
    int32_t N, H, dk, dv, dtype, chunk;
    int64_t T;
    bool scalar_gate = false;   // g is [T, H] (one rate per head) instead of [T, H, dk]
};

// Arguments of one decode call after host validation.
struct DecodeArgs {
    const void *q, *k, *v;
    const float *g, *beta;
    float *S;
    void *o;
    int32_t B, H, dk, dv, dtype;
    const int32_t *slots = nullptr;   // pooled decode: state slot of each sequence
    int32_t P = 0;                    // pooled decode: number of slots
    bool scalar_gate = false;         // g is [B, H] instead of [B, H, dk]
};

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);
cudaError_t launch_prefill_simt(const PrefillArgs &a, cudaStream_t stream);
cudaError_t launch_prefill_tc(const PrefillArgs &a, void *workspace, cudaStream_t stream);
size_t prefill_tc_workspace_bytes(int32_t N, int64_t T, int32_t H);

// Size of the fixed scratch array behind kda_prefill_chunked_noalloc.
#define KDA_NOALLOC_SCRATCH_MIB 64
// Chunks per window that fit that scratch for N sequences and H heads
// (0: not even one chunk fits).
int64_t noalloc_window_chunks(int32_t N, int32_t H);
cudaError_t launch_prefill_tc_noalloc(const PrefillArgs &a, cudaStream_t stream);
// Device status word of the fixed scratch on the current device (the caller
// has synchronised): nonzero when a bounded wait of the last no-allocation
// prefill on this device gave up.
cudaError_t noalloc_status(int32_t *word);

// Forced-timeout hook of the fault-injection test build (compiled with
// KDA_FAULT_INJECTION; absent from the library itself): while it is set, the
// per-chunk kernel of every tensor-core prefill waits on an mbarrier that
// nothing arrives at, before it issues any copy or tensor-core operation,
// gives up after a few iterations and reports KDA_ERR_TIMEOUT.
int fault_force_timeout();
// Prefill from host memory: q, k, v, g, beta, S0, o and S_T of `args` are
// host pointers, cu_seqlens of `args` is unused; `cu_host` holds the
// validated offsets in host memory.
struct HostPrefillArgs {
    PrefillArgs args;
    const int32_t *cu_host;
};
uint64_t prefill_host_workspace_bytes(int32_t N, int64_t T, int32_t H, int32_t dk, int32_t dv,
                                      int32_t dtype);
cudaError_t launch_prefill_host(const HostPrefillArgs &h, void *workspace, cudaStream_t stream);

// ---- element access helpers ------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Four consecutive elements starting at a 4-element-aligned index.
__device__ __forceinline__ float4 load4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    uint2 raw = *reinterpret_cast<const uint2 *>(p);
    __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162 *>(&raw.x);
    __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162 *>(&raw.y);
    float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void store4(float *p, float4 x) {
    *reinterpret_cast<float4 *>(p) = x;
}
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 x) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
    uint2 raw;
    raw.x = *reinterpret_cast<uint32_t *>(&lo);
    raw.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = raw;
}

// Sequence bounds read from device offsets, clamped into [0, T] so that
// inconsistent offsets never lead outside the token arrays.
__device__ __forceinline__ void seq_bounds(const int32_t *cu, int n, int64_t T,
                                           int64_t &bos, int64_t &eos) {
    int64_t a = cu[n], b = cu[n + 1];
    a = a < 0 ? 0 : (a > T ? T : a);
    b = b < a ? a : (b > T ? T : b);
    bos = a;
    eos = b;
}

}  // namespace kda
