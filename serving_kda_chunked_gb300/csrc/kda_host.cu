// kda_host.cu -- prefill from host memory (kda_prefill_chunked_host in kda.h).
//
// The token range is cut into pieces of 512 to 16 K tokens.  Each
// piece's inputs are copied into one of two device staging slots on a copy
// stream, the piece runs as an ordinary packed prefill on the caller's stream
// (the states of its sequences carried in a device state buffer, read and
// written in place), and its outputs go back on a second copy stream.  The
// host->device copies of piece p+1, the kernels of piece p and the
// device->host copy of piece p-1 therefore overlap; the host link is the
// bound (the whole call costs about the input copy plus one piece).
//
// Piece boundaries fall on chunk boundaries of the sequence they cut (a
// multiple of 64 tokens from its start), so every chunk is the same chunk as
// in a single call over the whole batch and only the state crosses pieces,
// in fp32 through the state buffer, as it crosses windows inside one call.
#include <mutex>
#include <vector>

#include "../../include/kda.h"
#include "kda_internal.cuh"
#include "kda_prefill_tc.cuh"

namespace kda {

namespace {

// Workspace of the tensor-core prefill for any call of at most N sequences
// and T tokens (a piece): the operand images grow with N and T; the segment
// maps of the chunk-affine scan (one sequence only) are taken at their
// largest segment count (the limit the scan plan of the tensor-core prefill
// uses), which is not monotone in T.
size_t prefill_tc_piece_workspace_bytes(int32_t N, int64_t T, int32_t H) {
    using namespace tcp;
    const int64_t bound = (T + C - 1) / C + N;
    const int64_t wch = bound < WINDOW_CHUNKS ? bound : WINDOW_CHUNKS;
    const size_t images = (size_t)ws_images_offset(N) + (size_t)wch * (size_t)H * CH_STRIDE;
    const int64_t gmax = H > 0 ? (128 / H + 4) / 8 : 0;
    const size_t maps = gmax >= 4 ? (size_t)H * gmax * 3 * (D * D * sizeof(float)) : 0;
    return ((images + 255) & ~(size_t)255) + maps;
}

// Each host->device copy carries a fixed cost of ~3 us on top of the link
// time (211 GB/s measured from pinned memory), and the last piece's kernels
// and output copy are not overlapped.  A call of 8 K tokens measured, per
// call: equal pieces, 16: 1.99 ms, 8: 1.93 ms, 4: 1.94 ms; with the pieces
// halving toward the end (down to 256 tokens), 12: 1.95 ms, 8: 1.91 ms,
// 6: 1.89 ms.  The copies alone, as one piece, take 1.70 ms.  Alternating
// the pieces over two copy streams measured slower (2.06 ms for 16 pieces).
constexpr int64_t PIECES = 6;         // full-size pieces per call (before the limits below)
constexpr int64_t PIECE_MIN = 512;    // tokens: keeps every SM busy in the per-chunk kernel
constexpr int64_t PIECE_MAX = 16384;  // tokens: bounds the staging buffers
constexpr int64_t CHUNK = 64;
constexpr int64_t TAIL_MIN = 256;     // tokens: the smallest piece at the end of a call

inline uint64_t align256(uint64_t x) { return (x + 255) & ~(uint64_t)255; }

// Tokens per piece for a call of T tokens (a multiple of 64, or T itself).
int64_t piece_cap(int64_t T) {
    int64_t p = (T + PIECES - 1) / PIECES;
    p = (p + CHUNK - 1) / CHUNK * CHUNK;
    if (p < PIECE_MIN) p = PIECE_MIN;
    if (p > PIECE_MAX) p = PIECE_MAX;
    return p < T ? p : T;
}

// Byte layout of the host-path workspace.
struct HostLayout {
    int64_t cap;                        // tokens per piece at most
    uint64_t tok_q, tok_k, tok_v, tok_g, tok_b, tok_o;   // bytes per token
    uint64_t pre, state, cu, cup, in[2], out[2], total;  // region offsets
    uint64_t in_k, in_v, in_g, in_b;    // offsets inside an input slot
};

HostLayout host_layout(int32_t N, int64_t T, int32_t H, int32_t dk, int32_t dv,
                       int32_t dtype) {
    HostLayout L;
    const uint64_t es = dtype == KDA_BF16 ? 2 : 4;
    L.cap = piece_cap(T);
    L.tok_q = (uint64_t)H * dk * es;
    L.tok_k = L.tok_q;
    L.tok_v = (uint64_t)H * dv * es;
    L.tok_g = (uint64_t)H * dk * 4;
    L.tok_b = (uint64_t)H * 4;
    L.tok_o = L.tok_v;
    const uint64_t c = (uint64_t)L.cap;
    L.in_k = align256(c * L.tok_q);
    L.in_v = L.in_k + align256(c * L.tok_k);
    L.in_g = L.in_v + align256(c * L.tok_v);
    L.in_b = L.in_g + align256(c * L.tok_g);
    const uint64_t slot_in = L.in_b + align256(c * L.tok_b);
    const uint64_t slot_out = align256(c * L.tok_o);
    const bool tensor_path = dtype == KDA_BF16 && dk == 128;
    L.pre = 256;   // word 0: the call's sticky device status
    uint64_t off = L.pre + (tensor_path ? align256(prefill_tc_piece_workspace_bytes(N, L.cap, H)) : 0);
    L.state = off; off += align256((uint64_t)N * H * dk * dv * 4);
    L.cu = off;    off += align256((uint64_t)(N + 1) * 4);
    L.cup = off;   off += align256((uint64_t)(N + 1) * 4);
    for (int s = 0; s < 2; ++s) { L.in[s] = off; off += slot_in; }
    for (int s = 0; s < 2; ++s) { L.out[s] = off; off += slot_out; }
    L.total = off;
    return L;
}

struct Piece {
    int64_t a, b;   // tokens [a, b)
    int32_t n0, n;  // sequences n0 .. n0 + n - 1 overlap it
};

// Cut [0, T) into pieces of at most `cap` tokens (at least TAIL_MIN, or what
// is left), each boundary on a chunk boundary of the sequence it falls in.  `cu` is validated (cu[0] = 0,
// non-decreasing, cu[N] = T).
std::vector<Piece> plan_pieces(const int32_t *cu, int32_t N, int64_t T, int64_t cap) {
    std::vector<Piece> out;
    int32_t m = 0;   // sequence containing token a (or the first with cu[m+1] > a)
    for (int64_t a = 0; a < T;) {
        // toward the end the pieces halve (down to TAIL_MIN tokens): the last
        // piece's kernels and output copy are the part of the call that
        // nothing overlaps
        const int64_t rem = T - a;
        int64_t len = (rem / 2 + CHUNK - 1) / CHUNK * CHUNK;
        if (len < TAIL_MIN) len = TAIL_MIN;
        if (rem - len < TAIL_MIN) len = rem;   // no piece smaller than TAIL_MIN after this one
        if (len > cap) len = cap;
        int64_t b = a + len;
        if (b >= T) {
            b = T;
        } else {
            int32_t j = m;
            while ((int64_t)cu[j + 1] <= b) ++j;      // cu[j] <= b < cu[j+1]
            const int64_t bos = cu[j];
            b = bos + (b - bos) / CHUNK * CHUNK;      // > a: see below
        }
        // b > a: if b stayed in a's sequence it moved down by less than 64 from
        // a + len >= a + 64 (a is on that sequence's chunk grid); otherwise it
        // is at least the start of a later sequence, which is > a.
        while ((int64_t)cu[m + 1] <= a) ++m;
        int32_t last = m;
        while (last + 1 < N && (int64_t)cu[last + 1] < b) ++last;
        out.push_back(Piece{a, b, m, last - m + 1});
        a = b;
    }
    return out;
}

// Offsets of the sequences n0 .. n0 + n - 1 clipped to the piece [a, b) and
// shifted to its start; thread 0 also keeps the first nonzero status that a
// piece's kernels left in their workspace word (`prev`), in the call's word.
__global__ void piece_offsets_kernel(const int32_t *__restrict__ cu, int n0, int n, int64_t a,
                                     int64_t b, int32_t *__restrict__ cup,
                                     const int32_t *prev, int32_t *sticky, int first) {
    if (threadIdx.x == 0) {
        if (first) *sticky = 0;
        else if (prev && *prev != 0 && *sticky == 0) *sticky = *prev;
    }
    if (n <= 0) return;   // status only
    for (int i = threadIdx.x; i <= n; i += blockDim.x) {
        int64_t x = cu[n0 + i];
        x = x < a ? a : (x > b ? b : x);
        cup[i] = (int32_t)(x - a);
    }
}

// Two copy streams and the events that order them, per device, created on
// first use.  Each device's mutex is held while a call enqueues its work on
// that device, so that concurrent calls never interleave their use of the
// events; calls on different devices do not wait for each other.
struct Lanes {
    std::mutex mu;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr, ready = nullptr;
    cudaEvent_t in[2] = {nullptr, nullptr}, comp[2] = {nullptr, nullptr},
                out[2] = {nullptr, nullptr};
};
Lanes g_lanes[64];

// (called with g_lanes[dev].mu held)
cudaError_t get_lanes(int dev, Lanes **out) {
    Lanes &L = g_lanes[dev];
    if (!L.h2d) {
        cudaError_t e = cudaStreamCreateWithFlags(&L.h2d, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&L.d2h, cudaStreamNonBlocking);
        cudaEvent_t *evs[] = {&L.start, &L.done, &L.ready, &L.in[0], &L.in[1], &L.comp[0],
                              &L.comp[1], &L.out[0], &L.out[1]};
        for (cudaEvent_t *ev : evs)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
    }
    *out = &L;
    return cudaSuccess;
}

}  // namespace

uint64_t prefill_host_workspace_bytes(int32_t N, int64_t T, int32_t H, int32_t dk, int32_t dv,
                                      int32_t dtype) {
    return host_layout(N, T, H, dk, dv, dtype).total;
}

cudaError_t launch_prefill_host(const HostPrefillArgs &h, void *workspace, cudaStream_t st) {
    const PrefillArgs &a = h.args;
    const HostLayout L = host_layout(a.N, a.T, a.H, a.dk, a.dv, a.dtype);
    const bool tensor_path = a.dtype == KDA_BF16 && a.dk == 128;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *sticky = reinterpret_cast<int32_t *>(ws);
    uint8_t *pre = ws + L.pre;
    float *state = reinterpret_cast<float *>(ws + L.state);
    int32_t *cu_d = reinterpret_cast<int32_t *>(ws + L.cu);
    int32_t *cup = reinterpret_cast<int32_t *>(ws + L.cup);
    const uint64_t state_row = (uint64_t)a.H * a.dk * a.dv;   // floats per sequence
    const uint64_t state_bytes = (uint64_t)a.N * state_row * 4;
    const std::vector<Piece> plan = plan_pieces(h.cu_host, a.N, a.T, L.cap);

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_lanes[dev].mu);
    Lanes *ln = nullptr;
    if ((e = get_lanes(dev, &ln)) != cudaSuccess) return e;

#define KDA_TRY(x) do { if ((e = (x)) != cudaSuccess) return e; } while (0)
    KDA_TRY(cudaEventRecord(ln->start, st));
    KDA_TRY(cudaStreamWaitEvent(ln->h2d, ln->start, 0));
    KDA_TRY(cudaStreamWaitEvent(ln->d2h, ln->start, 0));
    KDA_TRY(cudaMemcpyAsync(cu_d, h.cu_host, (size_t)(a.N + 1) * 4, cudaMemcpyHostToDevice, ln->h2d));
    if (a.S0)
        KDA_TRY(cudaMemcpyAsync(state, a.S0, state_bytes, cudaMemcpyHostToDevice, ln->h2d));
    else
        KDA_TRY(cudaMemsetAsync(state, 0, state_bytes, st));
    KDA_TRY(cudaEventRecord(ln->ready, ln->h2d));
    KDA_TRY(cudaStreamWaitEvent(st, ln->ready, 0));   // offsets and states are in place
    piece_offsets_kernel<<<1, 32, 0, st>>>(cu_d, 0, 0, 0, 0, cup, nullptr, sticky, 1);
    KDA_TRY(cudaGetLastError());

    const char *q_h = static_cast<const char *>(a.q), *k_h = static_cast<const char *>(a.k);
    const char *v_h = static_cast<const char *>(a.v);
    const char *g_h = reinterpret_cast<const char *>(a.g);
    const char *b_h = reinterpret_cast<const char *>(a.beta);
    char *o_h = static_cast<char *>(a.o);
    for (size_t p = 0; p < plan.size(); ++p) {
        const Piece &pc = plan[p];
        const int s = (int)(p & 1);
        const uint64_t nt = (uint64_t)(pc.b - pc.a);
        uint8_t *in = ws + L.in[s];
        uint8_t *out = ws + L.out[s];
        // inputs of piece p into slot s, once piece p - 2 is done with it
        if (p >= 2) KDA_TRY(cudaStreamWaitEvent(ln->h2d, ln->comp[s], 0));
        KDA_TRY(cudaMemcpyAsync(in, q_h + pc.a * L.tok_q, nt * L.tok_q, cudaMemcpyHostToDevice, ln->h2d));
        KDA_TRY(cudaMemcpyAsync(in + L.in_k, k_h + pc.a * L.tok_k, nt * L.tok_k, cudaMemcpyHostToDevice, ln->h2d));
        KDA_TRY(cudaMemcpyAsync(in + L.in_v, v_h + pc.a * L.tok_v, nt * L.tok_v, cudaMemcpyHostToDevice, ln->h2d));
        KDA_TRY(cudaMemcpyAsync(in + L.in_g, g_h + pc.a * L.tok_g, nt * L.tok_g, cudaMemcpyHostToDevice, ln->h2d));
        KDA_TRY(cudaMemcpyAsync(in + L.in_b, b_h + pc.a * L.tok_b, nt * L.tok_b, cudaMemcpyHostToDevice, ln->h2d));
        KDA_TRY(cudaEventRecord(ln->in[s], ln->h2d));
        // the piece's kernels, once its inputs are in and slot s's outputs of
        // piece p - 2 have left
        KDA_TRY(cudaStreamWaitEvent(st, ln->in[s], 0));
        if (p >= 2) KDA_TRY(cudaStreamWaitEvent(st, ln->out[s], 0));
        // (the status word of the previous piece: before piece 0 it holds
        // whatever the workspace held)
        piece_offsets_kernel<<<1, 256, 0, st>>>(cu_d, pc.n0, pc.n, pc.a, pc.b, cup,
                                                tensor_path && p > 0 ? reinterpret_cast<int32_t *>(pre) : nullptr,
                                                sticky, 0);
        KDA_TRY(cudaGetLastError());
        PrefillArgs pa = a;
        pa.q = in; pa.k = in + L.in_k; pa.v = in + L.in_v;
        pa.g = reinterpret_cast<const float *>(in + L.in_g);
        pa.beta = reinterpret_cast<const float *>(in + L.in_b);
        pa.S0 = state + (uint64_t)pc.n0 * state_row;
        pa.S_T = state + (uint64_t)pc.n0 * state_row;
        pa.cu_seqlens = cup;
        pa.N = pc.n;
        pa.T = (int64_t)nt;
        pa.o = out;
        KDA_TRY(tensor_path ? launch_prefill_tc(pa, pre, st) : launch_prefill_simt(pa, st));
        KDA_TRY(cudaEventRecord(ln->comp[s], st));
        // its outputs back to the host
        KDA_TRY(cudaStreamWaitEvent(ln->d2h, ln->comp[s], 0));
        KDA_TRY(cudaMemcpyAsync(o_h + pc.a * L.tok_o, out, nt * L.tok_o, cudaMemcpyDeviceToHost, ln->d2h));
        KDA_TRY(cudaEventRecord(ln->out[s], ln->d2h));
    }
    // fold the last piece's status, then the final states to the host
    piece_offsets_kernel<<<1, 32, 0, st>>>(cu_d, 0, 0, 0, 0, cup,
                                           tensor_path && !plan.empty() ? reinterpret_cast<int32_t *>(pre) : nullptr,
                                           sticky, 0);
    KDA_TRY(cudaGetLastError());
    KDA_TRY(cudaEventRecord(ln->ready, st));
    KDA_TRY(cudaStreamWaitEvent(ln->d2h, ln->ready, 0));
    KDA_TRY(cudaMemcpyAsync(a.S_T, state, state_bytes, cudaMemcpyDeviceToHost, ln->d2h));
    KDA_TRY(cudaEventRecord(ln->done, ln->d2h));
    KDA_TRY(cudaStreamWaitEvent(st, ln->done, 0));
#undef KDA_TRY
    return cudaSuccess;
}

}  // namespace kda
