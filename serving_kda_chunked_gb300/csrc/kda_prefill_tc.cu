// kda_prefill_tc.cu -- host side of the tensor-core prefill: tensor maps,
// workspace sizing, the chunk-affine scan plan and the kernel launches
// (layouts and the method overview in kda_prefill_tc.cuh).
#include "kda_prefill_tc.cuh"

#include <atomic>
#include <mutex>

namespace kda {
namespace tcp {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 3D map over a token-major [T][H][128] tensor; one box = 64 tokens of one
// head by 128 bytes of channels (64 bf16 or 32 fp32), landing with the
// 128-byte swizzle (16-byte chunk c of token row t at chunk c ^ (t % 8)).
bool token_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, uint32_t esize, int H,
               int64_t T) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)H * D * esize};
    cuuint32_t box[3] = {128u / esize, 1, (cuuint32_t)C};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device setup, once per device: the kernels' shared-memory limits (a
// function attribute of the device's context) and the SM count.
cudaError_t device_setup(int *nsm) {
    static std::mutex mu;
    static int sms[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!sms[dev]) {
        e = cudaFuncSetAttribute(intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)S1_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)S2_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(chain_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)S2W_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(segment_combine_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)COMB_BYTES);
        int n = 0;
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        sms[dev] = n > 0 ? n : 1;
    }
    *nsm = sms[dev];
    return cudaSuccess;
}

}  // namespace tcp

using namespace tcp;

namespace {

// Chunk-affine scan plan for one sequence of `chunks` chunks and H heads.
// The state chain of a (head, 32-column slice) is latency-bound, so when the
// 4 H slice chains leave most SMs idle, the chunks are cut into segments:
// phase 0 runs 4 + 8 (nseg - 1) chains per head, each over one segment (the
// segment maps), a short combine step chains their start states, and phase 1
// reruns segments 1.. (4 (nseg - 1) chains per head) for their outputs.  The
// chain latency falls from `chunks` steps to about 2 chunks / nseg.  nseg is
// held to (8 nseg - 4) H <= 128 so that phase 0 runs in one wave, and
// segments keep at least 16 chunks; with fewer than 4 segments it is off.
struct SegPlan { int nseg, seg_len; };
SegPlan segment_plan(int32_t N, int32_t H, int64_t chunks) {
    SegPlan pl{0, 0};
    if (N != 1 || H <= 0) return pl;
    const int64_t gmax = (128 / H + 4) / 8;
    if (gmax < 4 || chunks < 4 * 16) return pl;
    int64_t seg_len = (chunks + gmax - 1) / gmax;
    if (seg_len < 16) seg_len = 16;
    const int64_t nseg = (chunks + seg_len - 1) / seg_len;
    if (nseg < 4) return pl;
    pl.nseg = (int)nseg;
    pl.seg_len = (int)seg_len;
    return pl;
}

// bytes of segment maps for a window of `wch` chunks (0 when the scan is off)
size_t smaps_bytes(int32_t N, int32_t H, int64_t wch) {
    const SegPlan pl = segment_plan(N, H, wch);
    return pl.nseg ? (size_t)H * pl.nseg * 3 * (D * D * sizeof(float)) : 0;
}

}  // namespace

size_t prefill_tc_workspace_bytes(int32_t N, int64_t T, int32_t H) {
    const int64_t bound = (T + C - 1) / C + N;
    const int64_t wch = bound < WINDOW_CHUNKS ? bound : WINDOW_CHUNKS;
    const size_t images = (size_t)ws_images_offset(N) + (size_t)wch * (size_t)H * CH_STRIDE;
    const size_t maps = smaps_bytes(N, H, wch);
    return maps ? ((images + 255) & ~(size_t)255) + maps : images;
}

namespace {

// The prefill with windows of `window` chunks; `workspace` holds at least
// ws_images_offset(N) + window * H * CH_STRIDE bytes, plus (when `scan`) the
// segment maps of the chunk-affine scan behind them.
cudaError_t run_prefill_tc(const PrefillArgs &a, uint8_t *ws, int64_t window, bool scan,
                           cudaStream_t st) {
    int nsm = 1;
    cudaError_t e = device_setup(&nsm);
    if (e != cudaSuccess) return e;
    float *smaps = nullptr;
    if (scan) {
        const size_t images = (size_t)ws_images_offset(a.N) + (size_t)window * (size_t)a.H * CH_STRIDE;
        smaps = reinterpret_cast<float *>(ws + ((images + 255) & ~(size_t)255));
    }
    int32_t *hdr = reinterpret_cast<int32_t *>(ws);
    const int64_t bound = (a.T + C - 1) / C + a.N;
    int32_t *chunk_base = reinterpret_cast<int32_t *>(ws + WS_HEADER);
    chunk_table_kernel<<<1, 1024, 0, st>>>(a.cu_seqlens, a.N, a.T, (int)bound, hdr, chunk_base);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    K1Params p1;
    if (a.T > 0) {
        if (!token_map(&p1.tm_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.H, a.T) ||
            !token_map(&p1.tm_k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.H, a.T) ||
            !token_map(&p1.tm_v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.H, a.T))
            return cudaErrorInvalidValue;
        if (!a.scalar_gate &&
            !token_map(&p1.tm_g, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.H, a.T))
            return cudaErrorInvalidValue;
    }
    p1.g = a.g; p1.scalar_gate = a.scalar_gate ? 1 : 0;
    p1.force_timeout = fault_force_timeout();
    p1.beta = a.beta; p1.cu = a.cu_seqlens; p1.ws = ws; p1.N = a.N; p1.H = a.H; p1.T = a.T;
    for (int64_t w0 = 0; w0 < bound; w0 += window) {
        const int64_t w1 = w0 + window;
        p1.w0 = (int)w0; p1.w1 = (int)w1; p1.img0 = (int)w0;
        const int64_t wch = (bound - w0) < window ? (bound - w0) : window;
        K2Params p2;
        p2.S0 = a.S0; p2.S_T = a.S_T; p2.o = (__nv_bfloat16 *)a.o; p2.cu = a.cu_seqlens;
        p2.ws = ws; p2.N = a.N; p2.H = a.H; p2.T = a.T; p2.w0 = (int)w0; p2.w1 = (int)w1;
        p2.img0 = (int)w0;
        p2.nseg = 0; p2.seg_len = 0; p2.phase = 0; p2.smaps = smaps; p2.plan = nullptr;
        const SegPlan pl = smaps ? segment_plan(a.N, a.H, wch) : SegPlan{0, 0};
        if (a.T > 0) {
            const int64_t tasks = (w1 - w0) * a.H;
            const int g1 = (int)(tasks < nsm ? tasks : nsm);
            // a programmatic dependent of the kernel before it (the chunk
            // table, or the previous window's chain, which allows no early
            // launch): its setup overlaps the chunk table
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)g1);
            cfg.blockDim = dim3(K1_THREADS);
            cfg.dynamicSmemBytes = S1_BYTES;
            cfg.stream = st;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, intra_kernel, p1);
            if (e != cudaSuccess) return e;
        }
        if (pl.nseg) {            // chunk-affine scan over this window
            p2.nseg = pl.nseg; p2.seg_len = pl.seg_len; p2.phase = 0;
            chain_kernel<<<(unsigned)(a.H * (4 + 8 * (pl.nseg - 1))), K2_THREADS, S2_BYTES, st>>>(p2);
            segment_combine_kernel<<<(unsigned)(a.H * NSLICE), COMB_THREADS, COMB_BYTES, st>>>(
                smaps, pl.nseg);
            p2.phase = 1;
            chain_kernel<<<(unsigned)(a.H * 4 * (pl.nseg - 1)), K2_THREADS, S2_BYTES, st>>>(p2);
            e = cudaGetLastError();
            if (e != cudaSuccess) return e;
            continue;
        }
        // A chain is latency-bound: one (sequence, head, 32-column slice) per
        // SM finishes soonest when all slices run at once; with more than two
        // waves of slices, one CTA per (sequence, head) carrying all four
        // slices gets through about twice the chains per SM.  With that many
        // sequences, which of them have chunks in this window is known on the
        // device only: a one-block kernel lists them (longest chain first) and
        // picks the form, both forms are launched, and the CTAs of the form
        // not picked return at once.
        const int64_t slices = (int64_t)a.N * a.H * NSLICE;
        if (slices > 2 * (int64_t)nsm) {
            int32_t *plan = reinterpret_cast<int32_t *>(ws + ws_plan_offset(a.N));
            window_plan_kernel<<<1, 1024, 0, st>>>(chunk_base, a.N, (int)w0, (int)w1, a.H,
                                                   2 * nsm, plan);
            p2.plan = plan;
            chain_wide_kernel<<<(unsigned)((int64_t)a.N * a.H), K2W_THREADS, S2W_BYTES, st>>>(p2);
            chain_kernel<<<(unsigned)(2 * nsm), K2_THREADS, S2_BYTES, st>>>(p2);
        } else if (a.T > 0) {
            // right behind the per-chunk kernel: launched as its programmatic
            // dependent, so that its CTAs take the SMs the per-chunk kernel
            // frees while that kernel's last CTAs still run; they wait for
            // its completion (griddepcontrol.wait) before their first global
            // read of anything this call wrote
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)slices);
            cfg.blockDim = dim3(K2_THREADS);
            cfg.dynamicSmemBytes = S2_BYTES;
            cfg.stream = st;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, chain_kernel, p2);
            if (e != cudaSuccess) return e;
        } else {
            chain_kernel<<<(unsigned)slices, K2_THREADS, S2_BYTES, st>>>(p2);
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Fixed scratch for callers that cannot allocate device memory.  Every GPU
// that loads this library holds it until the process exits; all calls of
// the no-allocation entry point share it.
constexpr size_t NOALLOC_BYTES = (size_t)KDA_NOALLOC_SCRATCH_MIB << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_BYTES];

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs &a, void *workspace, cudaStream_t st) {
    const int64_t bound = (a.T + C - 1) / C + a.N;
    const int64_t window = bound < WINDOW_CHUNKS ? bound : WINDOW_CHUNKS;
    return run_prefill_tc(a, static_cast<uint8_t *>(workspace), window,
                          smaps_bytes(a.N, a.H, window) > 0, st);
}

int64_t noalloc_window_chunks(int32_t N, int32_t H) {
    const uint64_t head = ws_images_offset(N);
    if (head >= NOALLOC_BYTES) return 0;
    const uint64_t w = (NOALLOC_BYTES - head) / ((uint64_t)H * CH_STRIDE);
    return (int64_t)(w < (uint64_t)WINDOW_CHUNKS ? w : (uint64_t)WINDOW_CHUNKS);
}

namespace {
// Device address of the scratch array on the current device, looked up once
// per device with that device current (host code cannot use the symbol
// itself: it names a host-side stand-in).
cudaError_t noalloc_scratch(void **ws) {
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        e = cudaGetSymbolAddress(&addr[dev], g_noalloc_scratch);
        if (e != cudaSuccess) {
            addr[dev] = nullptr;
            return e;
        }
    }
    *ws = addr[dev];
    return cudaSuccess;
}
}  // namespace

cudaError_t launch_prefill_tc_noalloc(const PrefillArgs &a, cudaStream_t st) {
    void *ws = nullptr;
    cudaError_t e = noalloc_scratch(&ws);
    if (e != cudaSuccess) return e;
    const int64_t window = noalloc_window_chunks(a.N, a.H);
    if (window < 1) return cudaErrorInvalidValue;
    return run_prefill_tc(a, static_cast<uint8_t *>(ws), window, false, st);
}

cudaError_t noalloc_status(int32_t *word) {
    void *ws = nullptr;
    cudaError_t e = noalloc_scratch(&ws);
    if (e != cudaSuccess) return e;
    return cudaMemcpy(word, ws, sizeof *word, cudaMemcpyDeviceToHost);
}

#ifdef KDA_FAULT_INJECTION
static std::atomic<int> g_force_timeout{0};
int fault_force_timeout() { return g_force_timeout.load(); }
}  // namespace kda

// Test build only: switch the forced timeout on (nonzero) or off.
extern "C" void kda_test_force_timeout(int32_t on) { kda::g_force_timeout.store(on ? 1 : 0); }

namespace kda {
#else
int fault_force_timeout() { return 0; }
#endif

}  // namespace kda
