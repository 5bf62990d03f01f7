// kda_api.cu -- the C ABI: host-side validation and dispatch (see kda.h).
#include "../../include/kda.h"
#include "kda_internal.cuh"

#include <initializer_list>

namespace {

inline bool aligned16(const void *p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; }
inline bool aligned4(const void *p) { return p == nullptr || ((uintptr_t)p & 3u) == 0; }
inline bool head_ok(int32_t dk, int32_t dv) { return dk == dv && (dk == 64 || dk == 128); }

kda_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return KDA_OK;
    (void)cudaGetLastError();  // clear a sticky launch error for the caller
    return KDA_ERR_CUDA;
}

// The kernels run on the current device, so every buffer they touch must be
// memory that device owns (or managed memory).  Host memory -- page-locked
// memory is reachable from the device, but at PCIe/C2C speed -- and another
// device's memory are rejected before anything is launched.  Without a usable
// device the call fails with KDA_ERR_CUDA.
kda_status check_device_ptrs(std::initializer_list<const void *> ptrs) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    for (const void *p : ptrs) {
        if (!p) continue;
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
            (void)cudaGetLastError();
            return KDA_ERR_INVALID_ARG;
        }
        if (at.type == cudaMemoryTypeManaged) continue;
        if (at.type != cudaMemoryTypeDevice || at.device != dev) return KDA_ERR_INVALID_ARG;
    }
    return KDA_OK;
}

// Shared by the per-channel (KDA) and per-head (Gated DeltaNet) entry points,
// which differ only in the layout of g ([T, H, dk] vs [T, H]), and by the
// no-allocation entry point, which has no workspace argument.
kda_status prefill_impl(const void *q, const void *k, const void *v, const float *g,
                        const float *beta, const float *S0, const int32_t *cu_seqlens,
                        int32_t N, int64_t T_total, int32_t H, int32_t dk, int32_t dv,
                        int32_t dtype, int32_t chunk, void *o, float *S_T, void *workspace,
                        uint64_t workspace_bytes, bool scalar_gate, bool noalloc, void *stream) {
    if (N < 0 || T_total < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_FP32) return KDA_ERR_INVALID_ARG;
    if (dk <= 0 || dv <= 0 || chunk <= 0) return KDA_ERR_INVALID_ARG;
    if (!head_ok(dk, dv) || chunk != 64) return KDA_ERR_UNSUPPORTED;
    if (N == 0) return T_total == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    if (!cu_seqlens || !S_T) return KDA_ERR_INVALID_ARG;
    if (T_total > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !(scalar_gate ? aligned4(g) : aligned16(g)) ||
        !aligned16(o) || !aligned16(S0) || !aligned16(S_T) || !aligned4(beta) ||
        !aligned4(cu_seqlens))
        return KDA_ERR_INVALID_ARG;
    if ((int64_t)N * H * (dv / 32) > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
    const bool tensor_path = dtype == KDA_BF16 && dk == 128;
    if (tensor_path) {
        if (T_total / 64 + N > 0x3fffffffLL) return KDA_ERR_UNSUPPORTED;
        if (noalloc) {
            if (kda::noalloc_window_chunks(N, H) < 1) return KDA_ERR_TOO_LARGE;
        } else {
            const uint64_t need = kda::prefill_tc_workspace_bytes(N, T_total, H);
            if (!workspace || workspace_bytes < need || !aligned16(workspace))
                return KDA_ERR_INVALID_ARG;
        }
    }

    const kda_status dst = check_device_ptrs({q, k, v, g, beta, S0, cu_seqlens, o, S_T,
                                              tensor_path && !noalloc ? workspace : nullptr});
    if (dst != KDA_OK) return dst;

    kda::PrefillArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.S0 = S0;
    a.cu_seqlens = cu_seqlens; a.o = o; a.S_T = S_T;
    a.N = N; a.H = H; a.dk = dk; a.dv = dv; a.dtype = dtype; a.chunk = chunk;
    a.T = T_total;
    a.scalar_gate = scalar_gate;
    if (!tensor_path) return cuda_status(kda::launch_prefill_simt(a, (cudaStream_t)stream));
    if (noalloc) return cuda_status(kda::launch_prefill_tc_noalloc(a, (cudaStream_t)stream));
    return cuda_status(kda::launch_prefill_tc(a, workspace, (cudaStream_t)stream));
}

kda_status decode_impl(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, float *S, const int32_t *slots, int32_t P,
                       bool pooled, int32_t B, int32_t H, int32_t dk, int32_t dv, int32_t dtype,
                       void *o, bool scalar_gate, void *stream) {
    if (B < 0 || H <= 0 || (pooled && P <= 0)) return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_FP32) return KDA_ERR_INVALID_ARG;
    if (dk <= 0 || dv <= 0) return KDA_ERR_INVALID_ARG;
    if (!head_ok(dk, dv)) return KDA_ERR_UNSUPPORTED;
    if (B == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !S || !o || (pooled && !slots))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !(scalar_gate ? aligned4(g) : aligned16(g)) ||
        !aligned16(S) || !aligned16(o) || !aligned4(beta) || !aligned4(slots))
        return KDA_ERR_INVALID_ARG;
    if ((int64_t)B * H > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
    const kda_status dst = check_device_ptrs({q, k, v, g, beta, S, o, pooled ? slots : nullptr});
    if (dst != KDA_OK) return dst;

    kda::DecodeArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.S = S; a.o = o;
    a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.dtype = dtype;
    a.slots = pooled ? slots : nullptr; a.P = P;
    a.scalar_gate = scalar_gate;
    return cuda_status(kda::launch_decode(a, (cudaStream_t)stream));
}

}  // namespace

extern "C" {

kda_status kda_prefill_chunked(const void *q, const void *k, const void *v,
                               const float *g, const float *beta,
                               const float *S0, const int32_t *cu_seqlens,
                               int32_t N, int64_t T_total, int32_t H,
                               int32_t dk, int32_t dv, int32_t dtype,
                               int32_t chunk, void *o, float *S_T,
                               void *workspace, uint64_t workspace_bytes,
                               void *stream) {
    return prefill_impl(q, k, v, g, beta, S0, cu_seqlens, N, T_total, H, dk, dv, dtype, chunk,
                        o, S_T, workspace, workspace_bytes, false, false, stream);
}

kda_status kda_gdn_prefill_chunked(const void *q, const void *k, const void *v,
                                   const float *g, const float *beta,
                                   const float *S0, const int32_t *cu_seqlens,
                                   int32_t N, int64_t T_total, int32_t H,
                                   int32_t dk, int32_t dv, int32_t dtype,
                                   int32_t chunk, void *o, float *S_T,
                                   void *workspace, uint64_t workspace_bytes,
                                   void *stream) {
    return prefill_impl(q, k, v, g, beta, S0, cu_seqlens, N, T_total, H, dk, dv, dtype, chunk,
                        o, S_T, workspace, workspace_bytes, true, false, stream);
}

kda_status kda_prefill_chunked_noalloc(const void *q, const void *k, const void *v,
                                       const float *g, const float *beta,
                                       const float *S0, const int32_t *cu_seqlens,
                                       int32_t N, int64_t T_total, int32_t H,
                                       int32_t dk, int32_t dv, int32_t dtype,
                                       int32_t chunk, void *o, float *S_T,
                                       void *stream) {
    return prefill_impl(q, k, v, g, beta, S0, cu_seqlens, N, T_total, H, dk, dv, dtype, chunk,
                        o, S_T, nullptr, 0, false, true, stream);
}

kda_status kda_prefill_chunked_host(const void *q, const void *k, const void *v,
                                    const float *g, const float *beta,
                                    const float *S0, const int32_t *cu_seqlens,
                                    int32_t N, int64_t T_total, int32_t H,
                                    int32_t dk, int32_t dv, int32_t dtype,
                                    int32_t chunk, void *o, float *S_T,
                                    void *workspace, uint64_t workspace_bytes,
                                    void *stream) {
    if (N < 0 || T_total < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 && dtype != KDA_FP32) return KDA_ERR_INVALID_ARG;
    if (dk <= 0 || dv <= 0 || chunk <= 0) return KDA_ERR_INVALID_ARG;
    if (!head_ok(dk, dv) || chunk != 64) return KDA_ERR_UNSUPPORTED;
    if (N == 0) return T_total == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    if (T_total > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;   // offsets are int32
    if (!cu_seqlens || !S_T) return KDA_ERR_INVALID_ARG;
    if (T_total > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if ((int64_t)N * H * (dv / 32) > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
    const uint64_t need = kda::prefill_host_workspace_bytes(N, T_total, H, dk, dv, dtype);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return KDA_ERR_INVALID_ARG;
    // host buffers must not be device memory, the workspace must be (checked
    // where the runtime can tell)
    const void *host_ptrs[] = {cu_seqlens, q, k, v, g, beta, S0, o, S_T};
    for (const void *ptr : host_ptrs) {
        if (!ptr) continue;
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) { (void)cudaGetLastError(); continue; }
        if (at.type == cudaMemoryTypeDevice) return KDA_ERR_INVALID_ARG;
    }
    {
        cudaPointerAttributes at;
        int dev = -1;
        if (cudaPointerGetAttributes(&at, workspace) == cudaSuccess &&
            cudaGetDevice(&dev) == cudaSuccess) {
            if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
                return KDA_ERR_INVALID_ARG;
            if (at.type == cudaMemoryTypeDevice && at.device != dev)   // the call runs on the current device
                return KDA_ERR_INVALID_ARG;
        } else {
            (void)cudaGetLastError();
        }
    }
    // the offsets are read here: cu[0] = 0, non-decreasing, cu[N] = T_total
    if (cu_seqlens[0] != 0 || (int64_t)cu_seqlens[N] != T_total) return KDA_ERR_INVALID_ARG;
    for (int32_t n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return KDA_ERR_INVALID_ARG;

    kda::HostPrefillArgs h;
    kda::PrefillArgs &a = h.args;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.S0 = S0;
    a.cu_seqlens = nullptr; a.o = o; a.S_T = S_T;
    a.N = N; a.H = H; a.dk = dk; a.dv = dv; a.dtype = dtype; a.chunk = chunk;
    a.T = T_total;
    a.scalar_gate = false;
    h.cu_host = cu_seqlens;
    return cuda_status(kda::launch_prefill_host(h, workspace, (cudaStream_t)stream));
}

uint64_t kda_prefill_host_workspace_size(int32_t N, int64_t T_total, int32_t H, int32_t dk,
                                         int32_t dv, int32_t dtype, int32_t chunk) {
    if (N <= 0 || T_total < 0 || T_total > 0x7fffffffLL || H <= 0 || !head_ok(dk, dv) ||
        chunk != 64 || (dtype != KDA_BF16 && dtype != KDA_FP32))
        return 0;
    return kda::prefill_host_workspace_bytes(N, T_total, H, dk, dv, dtype);
}

uint64_t kda_noalloc_scratch_bytes(void) { return (uint64_t)KDA_NOALLOC_SCRATCH_MIB << 20; }

uint64_t kda_prefill_workspace_size(int32_t N, int64_t T_total, int32_t H, int32_t dk,
                                    int32_t dv, int32_t dtype, int32_t chunk) {
    if (N <= 0 || T_total < 0 || H <= 0 || !head_ok(dk, dv) || chunk != 64) return 0;
    if (dtype != KDA_BF16 || dk != 128) return 0;
    return (uint64_t)kda::prefill_tc_workspace_bytes(N, T_total, H);
}

kda_status kda_prefill_check(const void *workspace, void *stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_status(e);
    if (!workspace) return KDA_OK;
    int32_t word = 0;
    e = cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
    return word != 0 ? KDA_ERR_TIMEOUT : KDA_OK;
}

kda_status kda_prefill_noalloc_check(void *stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_status(e);
    int32_t word = 0;
    e = kda::noalloc_status(&word);
    if (e != cudaSuccess) return cuda_status(e);
    return word != 0 ? KDA_ERR_TIMEOUT : KDA_OK;
}

kda_status kda_decode_step(const void *q, const void *k, const void *v,
                           const float *g, const float *beta, float *S,
                           int32_t B, int32_t H, int32_t dk, int32_t dv,
                           int32_t dtype, void *o, void *stream) {
    return decode_impl(q, k, v, g, beta, S, nullptr, 0, false, B, H, dk, dv, dtype, o, false,
                       stream);
}

kda_status kda_gdn_decode_step(const void *q, const void *k, const void *v,
                               const float *g, const float *beta, float *S,
                               int32_t B, int32_t H, int32_t dk, int32_t dv,
                               int32_t dtype, void *o, void *stream) {
    return decode_impl(q, k, v, g, beta, S, nullptr, 0, false, B, H, dk, dv, dtype, o, true,
                       stream);
}

kda_status kda_decode_step_pooled(const void *q, const void *k, const void *v,
                                  const float *g, const float *beta, float *S_pool,
                                  const int32_t *slots, int32_t P, int32_t B, int32_t H,
                                  int32_t dk, int32_t dv, int32_t dtype, void *o,
                                  void *stream) {
    return decode_impl(q, k, v, g, beta, S_pool, slots, P, true, B, H, dk, dv, dtype, o, false,
                       stream);
}

kda_status kda_gdn_decode_step_pooled(const void *q, const void *k, const void *v,
                                      const float *g, const float *beta, float *S_pool,
                                      const int32_t *slots, int32_t P, int32_t B, int32_t H,
                                      int32_t dk, int32_t dv, int32_t dtype, void *o,
                                      void *stream) {
    return decode_impl(q, k, v, g, beta, S_pool, slots, P, true, B, H, dk, dv, dtype, o, true,
                       stream);
}

const char *kda_status_string(int32_t status) {
    switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: shape, chunk or dtype not supported";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA call failed";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded device wait gave up";
    case KDA_ERR_TOO_LARGE:
        return "KDA_ERR_TOO_LARGE: N or H too large for the fixed scratch of the no-allocation entry point";
    default: return "KDA_ERR_UNKNOWN: unknown status";
    }
}

int32_t kda_abi_version(void) { return (2 << 16) | 4; }

}  // extern "C"
