/*
 * kda.h -- C ABI of the KDA (Kimi Delta Attention) kernels for GB300 (sm_103a).
 *
 * KDA is a gated delta-rule linear attention with a per-channel gate.  Per
 * head it keeps a fixed-size state S (dk x dv, fp32) and, for every token t:
 *
 *     S   = Diag(exp(g_t)) S                decay first, one rate per channel
 *     S   = S + beta_t k_t (v_t - S^T k_t)^T   write the delta along k_t
 *     o_t = S^T q_t                          read out with the new state
 *
 * Sources: the delta rule and the decay-then-write order are in the lineage
 * essay "Baseten 엔지니어가 분석한 7년간의 어텐션 메커니즘 진화: GPT-2부터
 * Kimi K3까지", sections "DeltaNet: 이제 메모리를 편집할 수 있습니다" and
 * "Gated DeltaNet: 이제는 '망각'할 수 있습니다"; the per-channel gate in its
 * section "KDA: Kimi의 비법" and in "KV 캐시를 75% 줄였는데 성능은 더
 * 좋아졌다", section "KDA: 지우고 다시 쓰는 메모, 채널마다 다른 망각률".
 * The chunked form of prefill follows the essay's section "병렬화 트릭"
 * (chunks of C = 64 tokens, masked attention inside a chunk, the state
 * carried between chunks, a Householder/UT reparameterisation resolving all
 * deltas of a chunk at once).
 *
 * Conventions for every entry point
 *   - All tensors are dense, row-major, contiguous, in DEVICE memory owned by
 *     the caller.  Base pointers must be 16-byte aligned.  The library never
 *     allocates, frees or retains caller memory and keeps no per-call state.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL means
 *     the legacy default stream).  Outputs are valid once the stream reaches
 *     that point.
 *   - Arguments are validated on the host before any launch, without reading
 *     device memory.  A rejected call launches nothing and returns
 *     KDA_ERR_INVALID_ARG (malformed) or KDA_ERR_UNSUPPORTED (well formed but
 *     outside the compiled shapes).  A failed launch returns KDA_ERR_CUDA; the
 *     CUDA error is cleared with cudaGetLastError so that it does not leak
 *     into the caller's later checks.  No C++ exception or abort crosses the
 *     ABI.
 *   - Work runs on the CURRENT device (cudaGetDevice); `stream` must belong to
 *     it.  Every non-NULL tensor pointer of a device entry point is checked
 *     with cudaPointerGetAttributes: memory of another device, host memory
 *     (page-locked or not) and pointers the runtime does not know are
 *     rejected with KDA_ERR_INVALID_ARG; managed memory is accepted.  With no
 *     usable device the call returns KDA_ERR_CUDA.
 *   - The library caches per-device state for the life of the process
 *     (kernel attributes, the address of the no-allocation scratch, the
 *     host-buffer entry point's streams).  Do not use it across a
 *     cudaDeviceReset of a device it has run on.
 *   - Gates g are the log of the per-channel forgetting rate alpha in (0, 1]:
 *     finite values <= 0.  beta is the write strength in [0, 1].
 */
#ifndef KDA_H
#define KDA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* null pointer, misalignment, bad size       */
    KDA_ERR_UNSUPPORTED = 2,  /* head size / chunk / dtype not compiled in   */
    KDA_ERR_CUDA = 3,         /* a CUDA launch or attribute call failed      */
    KDA_ERR_TIMEOUT = 4,      /* a bounded device wait gave up (see check) */
    KDA_ERR_TOO_LARGE = 5     /* beyond the fixed scratch of the no-allocation
                                 entry point                                  */
} kda_status;

typedef enum kda_dtype {
    KDA_BF16 = 0,             /* q, k, v and o are bfloat16                  */
    KDA_FP32 = 1              /* q, k, v and o are float32                   */
} kda_dtype;

/*
 * kda_prefill_chunked -- chunked prefill over a packed batch of N sequences.
 *
 *   q, k       [T_total, H, dk]   dtype        queries, keys
 *   v          [T_total, H, dv]   dtype        values
 *   g          [T_total, H, dk]   float32      log-gate, finite, <= 0
 *   beta       [T_total, H]       float32      write strength
 *   S0         [N, H, dk, dv]     float32      initial states, or NULL (zeros)
 *   cu_seqlens [N + 1]            int32        sequence offsets: cu[0] = 0,
 *                                              non-decreasing, cu[N] = T_total
 *   o          [T_total, H, dv]   dtype        outputs (written)
 *   S_T        [N, H, dk, dv]     float32      final states (written); may be
 *                                              the same buffer as S0
 *   dk, dv     64 or 128, dk == dv
 *   chunk      64 (tokens per chunk); chunks never cross sequences and a
 *              partial last chunk is handled as if padded with no-op tokens
 *   dtype      KDA_BF16 or KDA_FP32
 *   workspace  device scratch of at least kda_prefill_workspace_size(...)
 *              bytes, 16-byte aligned, owned by the caller; may be NULL when
 *              that size is 0.  Its contents on entry do not matter; calls
 *              that share one workspace must not overlap on the GPU.
 *
 * With bf16 inputs and dk = dv = 128 the work runs on the tensor cores in two
 * kernels per window of up to 2048 chunks: one resolves every (chunk, head)
 * independently and writes its operands to the workspace, the next walks
 * each sequence's chunks in order carrying the fp32 state.  Every other case
 * (fp32 inputs, or dk = dv = 64) runs a CUDA-core kernel in fp32 arithmetic
 * that needs no workspace.
 *
 * Sequence n covers tokens [cu[n], cu[n+1]).  A sequence of length 0 copies
 * its S0 (or zeros) to S_T.  cu_seqlens lives in device memory and is not
 * read on the host; the kernels clamp every offset into [0, T_total], so
 * inconsistent offsets can only shorten sequences, never cause an
 * out-of-bounds access.  N = 0 with T_total = 0 is a valid no-op.
 */
kda_status kda_prefill_chunked(const void *q, const void *k, const void *v,
                               const float *g, const float *beta,
                               const float *S0, const int32_t *cu_seqlens,
                               int32_t N, int64_t T_total, int32_t H,
                               int32_t dk, int32_t dv, int32_t dtype,
                               int32_t chunk, void *o, float *S_T,
                               void *workspace, uint64_t workspace_bytes,
                               void *stream);

/*
 * Bytes of workspace kda_prefill_chunked needs for these sizes (0 for fp32
 * inputs).  Pure host arithmetic: no device access.  Returns 0 as well for
 * arguments that kda_prefill_chunked would reject.
 */
uint64_t kda_prefill_workspace_size(int32_t N, int64_t T_total, int32_t H,
                                    int32_t dk, int32_t dv, int32_t dtype,
                                    int32_t chunk);

/*
 * Synchronise `stream` and report the device-side status of the last
 * kda_prefill_chunked call that used `workspace`: KDA_ERR_TIMEOUT if one of
 * its kernels gave up on a bounded wait (its outputs are then incomplete: a
 * state-chain kernel that finds the per-chunk kernel of its window failed
 * writes nothing), KDA_ERR_CUDA if the stream reports an error, else KDA_OK.
 */
kda_status kda_prefill_check(const void *workspace, void *stream);

/*
 * kda_prefill_chunked_noalloc -- kda_prefill_chunked for callers that cannot
 * allocate device memory: same arguments, outputs and results, no workspace.
 * (This entry point has no counterpart in the method's description; it exists
 * for integration.)
 *
 * Some callers cannot call cudaMalloc or any allocating library routine: code
 * running while a CUDA graph is being built by someone else's allocator, a
 * host process whose device memory is owned by a framework, or plain-C
 * callers that hold only the tensors they were handed.  This variant keeps
 * its scratch in one fixed device array of kda_noalloc_scratch_bytes() bytes
 * (64 MiB) inside the library, held by every GPU that loads the library
 * until the process exits.  Long inputs are processed in as many windows of
 * chunks as that array needs; the call is rejected with KDA_ERR_TOO_LARGE
 * only when not even one chunk of all H heads (74,240 bytes each) plus a
 * header of 8 N + 268 bytes (the chunk table and the chain plan) fits.
 *
 * - The first call on a device looks up the array's device address with
 *   cudaGetSymbolAddress while that device is current; make that first call
 *   outside any stream capture.
 * - Every call on a device shares the array and leaves its contents behind;
 *   each call rewrites what it reads, so no clearing is needed, but calls that
 *   overlap on the GPU (other streams, other host threads) race on it.
 * - It calls no allocator: no cudaMalloc, cudaFree or allocating library
 *   routine.  fp32 and d = 64 inputs need no scratch at all.
 * - Its device-side status (a bounded wait that gave up) is kept in the first
 *   word of the array; kda_prefill_noalloc_check reads it.
 */
kda_status kda_prefill_chunked_noalloc(const void *q, const void *k, const void *v,
                                       const float *g, const float *beta,
                                       const float *S0, const int32_t *cu_seqlens,
                                       int32_t N, int64_t T_total, int32_t H,
                                       int32_t dk, int32_t dv, int32_t dtype,
                                       int32_t chunk, void *o, float *S_T,
                                       void *stream);

/* Size in bytes of the fixed scratch array behind the no-allocation entry. */
uint64_t kda_noalloc_scratch_bytes(void);

/*
 * kda_prefill_noalloc_check -- kda_prefill_check for the no-allocation entry
 * point: synchronise `stream`, then read the status word that the last
 * kda_prefill_chunked_noalloc call on the current device left in the fixed
 * scratch array.  KDA_ERR_TIMEOUT if one of its kernels gave up on a bounded
 * wait (its outputs were then left incomplete or untouched), KDA_ERR_CUDA if
 * the stream reports an error, else KDA_OK (also before any such call).  The
 * word is shared like the rest of the array: a no-allocation call enqueued on
 * another stream of the same device between that call and this check
 * overwrites it.  (No counterpart in the method's description.)
 */
kda_status kda_prefill_noalloc_check(void *stream);

/*
 * kda_prefill_chunked_host -- kda_prefill_chunked with the tensors in HOST
 * memory: the call copies the inputs in and the outputs out itself, and
 * overlaps those copies with the kernels.  (No counterpart in the method's
 * description; it serves callers whose activations live on the host.)
 *
 *   q, k, v, g, beta, S0, o, S_T   as kda_prefill_chunked, in host memory;
 *              page-locked memory (cudaHostAlloc, cudaHostRegister) lets the
 *              copies run asynchronously, pageable memory works but the
 *              runtime then stages each copy through the host
 *   cu_seqlens [N + 1] int32 in host memory, read by this call on the host:
 *              cu[0] = 0, non-decreasing, cu[N] = T_total, else
 *              KDA_ERR_INVALID_ARG (so T_total < 2^31)
 *   workspace  DEVICE scratch of at least kda_prefill_host_workspace_size(...)
 *              bytes, 16-byte aligned; calls sharing it must not overlap
 *
 * The token range is cut into pieces of about T_total / 6 tokens (at least
 * 512, at most 16,384) that halve toward the end of the call (down to 256
 * tokens), every cut on a 64-token chunk boundary of the sequence it falls
 * in.  Each piece is copied into one of two device staging slots,
 * runs as a packed prefill over the sequences it overlaps (their states
 * carried in a device state buffer in the workspace, exactly as the state
 * crosses windows inside one kda_prefill_chunked call), and its outputs are
 * copied back while the next piece is copied in and computed.  The results
 * equal those of kda_prefill_chunked on the same values.
 *
 * The copies run on two internal streams per device (created, with their
 * events, on the first call on that device and kept until the process ends);
 * the call is ordered after earlier work on `stream`, and `stream` reaches
 * its end only after the last copy into o and S_T.  Host buffers must stay
 * valid and unchanged (outputs: unread) until then.  Calls from several host
 * threads on one device are serialised while they enqueue; calls on different
 * devices are not.  With pageable (not page-locked) buffers each copy runs
 * synchronously with respect to the host, so the pieces no longer overlap
 * their copies with the kernels and the call takes about as long as its
 * copies plus its kernels in series.  kda_prefill_check(workspace,
 * stream) reports the device-side status of every piece.  Pointers that the
 * runtime identifies as device memory in place of a host buffer (or host
 * memory, or another device's memory, as the workspace) are rejected with
 * KDA_ERR_INVALID_ARG.  The call runs on the current device.
 */
kda_status kda_prefill_chunked_host(const void *q, const void *k, const void *v,
                                    const float *g, const float *beta,
                                    const float *S0, const int32_t *cu_seqlens,
                                    int32_t N, int64_t T_total, int32_t H,
                                    int32_t dk, int32_t dv, int32_t dtype,
                                    int32_t chunk, void *o, float *S_T,
                                    void *workspace, uint64_t workspace_bytes,
                                    void *stream);

/*
 * Bytes of device workspace kda_prefill_chunked_host needs for these sizes
 * (staging for two pieces, the prefill scratch of one piece, the N states and
 * the offsets).  Pure host arithmetic; 0 for arguments the call would reject
 * on their sizes alone (and for N = 0, which needs none).
 */
uint64_t kda_prefill_host_workspace_size(int32_t N, int64_t T_total, int32_t H,
                                         int32_t dk, int32_t dv, int32_t dtype,
                                         int32_t chunk);

/*
 * kda_decode_step -- one token for each of B independent sequences; the
 * states are updated in place.
 *
 *   q, k       [B, H, dk]         dtype
 *   v          [B, H, dv]         dtype
 *   g          [B, H, dk]         float32      log-gate, finite, <= 0
 *   beta       [B, H]             float32
 *   S          [B, H, dk, dv]     float32      read, then overwritten with S'
 *   o          [B, H, dv]         dtype        outputs (written)
 *   dk, dv     64 or 128, dk == dv
 *
 * The essay's section "KV 캐시: 재계산하지 말고 저장하라" notes that decode
 * is bound by memory bandwidth, not arithmetic: this kernel streams each
 * state from HBM once and writes it back once.  B = 0 is a valid no-op.
 * S must not overlap any input or output.
 */
kda_status kda_decode_step(const void *q, const void *k, const void *v,
                           const float *g, const float *beta, float *S,
                           int32_t B, int32_t H, int32_t dk, int32_t dv,
                           int32_t dtype, void *o, void *stream);

/*
 * kda_decode_step_pooled -- one decode token for each of B sequences whose
 * states live in a shared pool of P slots; slot slots[b] holds the state of
 * sequence b and is updated in place.
 *
 *   q, k       [B, H, dk]         dtype
 *   v          [B, H, dv]         dtype
 *   g          [B, H, dk]         float32      log-gate, finite, <= 0
 *   beta       [B, H]             float32
 *   S_pool     [P, H, dk, dv]     float32      slots named in `slots` are
 *                                              read and overwritten
 *   slots      [B]                int32        device memory; a value outside
 *                                              [0, P) skips that sequence:
 *                                              its o row is zeroed and no
 *                                              state is touched
 *   o          [B, H, dv]         dtype
 *
 * This is the serving form of decode: a KDA state has a fixed size however
 * long the context (the essay's section "선형 어텐션 (Linear Attention):
 * 고정된 크기의 메모리"), so concurrent sessions can each own one slot of a
 * preallocated pool instead of a growing KV cache (the explainer's section
 * "한국 개발자에게 주는 시사점": the number of concurrent requests is set
 * by how much cache memory is left).  The slots of the non-skipped sequences
 * must be distinct (two sequences in one slot race).  Slot values are not
 * read on the host.  B = 0 is a valid no-op.
 */
kda_status kda_decode_step_pooled(const void *q, const void *k, const void *v,
                                  const float *g, const float *beta, float *S_pool,
                                  const int32_t *slots, int32_t P, int32_t B, int32_t H,
                                  int32_t dk, int32_t dv, int32_t dtype, void *o,
                                  void *stream);

/*
 * kda_gdn_prefill_chunked, kda_gdn_decode_step -- the same two operations for
 * Gated DeltaNet, whose gate is one scalar per head and token instead of one
 * rate per channel.  The lineage essay's section "Gated DeltaNet: 이제는
 * '망각'할 수 있습니다" gives its update (decay the old memory by alpha, then
 * write the delta along k); its section "KDA: Kimi의 비법" states that KDA
 * differs from it only in turning that scalar alpha into a per-channel
 * vector.  So a Gated DeltaNet head is a KDA head whose dk gates are all equal,
 * and these entry points run the KDA kernels reading one gate per head:
 *
 *   g   [T_total, H]   (prefill)   or   [B, H]   (decode)   float32, log of
 *       alpha, finite, <= 0; 4-byte alignment suffices.
 *
 * Every other argument, the workspace (kda_prefill_workspace_size gives its
 * size here too), the outputs, the status codes and kda_prefill_check are as
 * for kda_prefill_chunked and kda_decode_step.
 */
kda_status kda_gdn_prefill_chunked(const void *q, const void *k, const void *v,
                                   const float *g, const float *beta,
                                   const float *S0, const int32_t *cu_seqlens,
                                   int32_t N, int64_t T_total, int32_t H,
                                   int32_t dk, int32_t dv, int32_t dtype,
                                   int32_t chunk, void *o, float *S_T,
                                   void *workspace, uint64_t workspace_bytes,
                                   void *stream);

kda_status kda_gdn_decode_step(const void *q, const void *k, const void *v,
                               const float *g, const float *beta, float *S,
                               int32_t B, int32_t H, int32_t dk, int32_t dv,
                               int32_t dtype, void *o, void *stream);

/* Gated DeltaNet decode over a state-slot pool: kda_decode_step_pooled with
 * one log-gate per head, g [B, H] float32 (4-byte alignment suffices). */
kda_status kda_gdn_decode_step_pooled(const void *q, const void *k, const void *v,
                                      const float *g, const float *beta, float *S_pool,
                                      const int32_t *slots, int32_t P, int32_t B, int32_t H,
                                      int32_t dk, int32_t dv, int32_t dtype, void *o,
                                      void *stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char *kda_status_string(int32_t status);

/* ABI version of this library: (major << 16) | minor. */
int32_t kda_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
