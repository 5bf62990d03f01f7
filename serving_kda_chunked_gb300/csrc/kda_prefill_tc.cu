// kda_prefill_tc.cu -- chunked KDA prefill on the 5th-generation tensor cores
// (tcgen05 + TMEM), bf16 inputs, fp32 state.
//
// Method: the chunkwise-parallel form of the lineage essay "GPT-2부터 Kimi
// K3까지", section "병렬화 트릭" -- chunks of C = 64 tokens, masked attention
// inside a chunk, the state plus a matmul between chunks, and the deltas of a
// chunk resolved at once through a UT (Householder-style) transform -- with
// the per-channel gate of its section "KDA: Kimi의 비법".  For a chunk with
// per-channel cumulative log-gate gamma and entering state S:
//
//   A[r,i] = beta_r sum_c k_rc k_ic e^(gamma_rc - gamma_ic)   i <  r
//   P[r,i] =        sum_c q_rc k_ic e^(gamma_rc - gamma_ic)   i <= r
//   T  = (I + A)^-1,  T' = T Diag(beta)
//   W  = T' (K * e^gamma),  U~ = T' V                      (independent of S)
//   U  = U~ - W S,   O = (Q * e^gamma) S + P U,
//   S <- Diag(e^gamma_last) S + (K * e^(gamma_last - gamma))^T U
//
// Two kernels split that along the only sequential dependency (the state):
//
//  * intra_kernel (K1) runs every (chunk, head) independently: the gate scan
//    and factors on CUDA cores, A and P on tcgen05 (tf32), the triangular
//    inverse on CUDA cores (fp32, 16x16 blocks), W and U~ on tcgen05 (fp16).
//    It writes the chunk's operands to a workspace, already laid out as the
//    shared-memory images the second kernel's MMAs read.
//  * chain_kernel (K2) walks the chunks of one (sequence, head, block of 32
//    state columns) in order with the fp32 state in registers: W S and Q^ S,
//    then K^T U and P U, each a tcgen05 round trip.  Operand images arrive
//    with bulk async copies, double buffered.  chain_wide_kernel is the same
//    walk for all 128 columns in one CTA (for batches with many chains); for
//    one sequence with few heads, the chunk-affine scan runs the slice chains
//    over segments and chains the segments' maps (segment_combine_kernel).
//
// Gate factors inside a chunk are referenced to the chunk start (K e^gamma,
// K e^-gamma), which stays inside fp32 while every channel's log-gate sum over
// the chunk is above -80; a chunk beyond that forms A and P pair by pair with
// e^(gamma_r - gamma_i) <= 1 instead, so any gate strength gives finite results.
//
// Operand precision (chosen with a CPU emulation against the fp64 oracle):
// A and P use tf32 operands (the gated factors need fp32 range); every other
// product uses fp16 operands with fp32 accumulation; the state stays fp32.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <mutex>

namespace kda {
namespace {

using namespace tc;

constexpr int C = 64;          // tokens per chunk
constexpr int D = 128;         // dk = dv
constexpr int DVS = 32;        // state columns per chain CTA
constexpr int NSLICE = D / DVS;

// workspace: header | chunk table | per (chunk, head) operand images
constexpr uint32_t WS_HEADER = 256;
constexpr uint32_t IMG_W = 0;          // W   [64 x 128] fp16, K-major SW128 (2 atoms)
constexpr uint32_t IMG_Q = 16384;      // Q^  [64 x 128] fp16, K-major SW128 (2 atoms)
constexpr uint32_t IMG_KT = 32768;     // Kb [64 x 128] fp16, [r][c] SW128 (MN-major A)
constexpr uint32_t IMG_P = 49152;      // P   [64 x 64] fp16, K-major SW128
constexpr uint32_t IMG_U = 57344;      // U~  [4 slices][64][32] fp16
constexpr uint32_t IMG_G = 73728;      // e^gamma_last [128] fp32
constexpr uint32_t CH_STRIDE = 74240;  // bytes per (chunk, head)
constexpr int WINDOW_CHUNKS = 2048;    // chunks per K1/K2 window

__host__ __device__ inline uint64_t ws_images_offset(int N) {
    uint64_t off = WS_HEADER + 4ull * (uint64_t)(N + 1);
    return (off + 1023) & ~1023ull;
}

// ------------------------------------------------------------------------------
// chunk table: chunk_base[n] = number of 64-token chunks before sequence n,
// capped at `cap` (the host's bound ceil(T/64) + N, which sizes the workspace):
// only overlapping, inconsistent offsets can reach the cap, and then the
// excess chunks are dropped instead of written past the workspace.
// ------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
chunk_table_kernel(const int32_t *__restrict__ cu, int N, int64_t T, int cap,
                   int32_t *ws_hdr, int32_t *chunk_base) {
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) { carry_s = 0; ws_hdr[0] = 0; }
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int n = base + tid;
        int cnt = 0;
        if (n < N) {
            int64_t bos, eos;
            seq_bounds(cu, n, T, bos, eos);
            cnt = (int)((eos - bos + C - 1) / C);
        }
        int x = cnt;   // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int t = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            warp_tot[lane] = t;   // inclusive over warps
        }
        __syncthreads();
        const int excl = x - cnt + (warp > 0 ? warp_tot[warp - 1] : 0);
        if (n < N) chunk_base[n] = min(carry_s + excl, cap);
        __syncthreads();
        if (tid == 0) carry_s += warp_tot[31];
        __syncthreads();
    }
    if (tid == 0) chunk_base[N] = min(carry_s, cap);
}

__device__ __forceinline__ void ws_fail(int32_t *ws_hdr, int code) { atomicExch(ws_hdr, code); }

// sequence holding global chunk c (chunk_base is non-decreasing)
__device__ __forceinline__ int find_seq(const int32_t *chunk_base, int N, int c) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_base[mid] <= c) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// ------------------------------------------------------------------------------
// K1: intra-chunk kernel
// ------------------------------------------------------------------------------
// One CTA per SM walks (chunk, head) tasks, chunk-major.  Per task:
//   1. TMA brings k, q, v (bf16) and g (fp32) rows [t0, t0 + 64) of head h
//      into staging; issued during the previous task, as soon as its prep
//      has consumed the staging tiles.
//   2. Per-channel cumulative log-gate (in place), e^gamma_last, range check;
//      the previous task's W/U MMA finishes underneath.
//   3. Element-wise prep, 8 channels of one row per unit: tf32 operands
//      [K e^g ; Q e^g] and K e^-g for A / P, fp16 K e^g and V for W / U~, the
//      Q^ and Kbar workspace images; the previous task's W and U~ leave TMEM
//      for the workspace in two rounds hidden behind it.
//   4. One M = 128 tf32 MMA group (warps 12-15 issue one channel atom each):
//      rows 0-63 give A / beta, rows 64-127 give P.  A chunk whose decay
//      exceeds e^80 on some channel would overflow those factors, so it takes
//      an exact pairwise CUDA-core path instead.
//   5. T = (I + A)^-1 on CUDA cores by warps 0-5 (fp32, 16 x 16 blocks,
//      register-tiled block forward substitution), written as the fp16 image
//      of T' = T Diag(beta).
//   6. W = T' (K e^g), U~ = T' V on tcgen05 (fp16), waited for in step 2 of
//      the next task.
constexpr int K1_THREADS = 512;
constexpr int K1_ISSUER0 = 12;  // warps 12-15 issue the A/P MMAs
constexpr uint32_t S1_STG_K = 0, S1_STG_Q = 16384, S1_STG_V = 32768;  // bf16 [64][128]
constexpr uint32_t S1_STG_G = 49152;                                  // fp32 [64][128]
constexpr uint32_t S1_OPA = 81920;    // tf32 [K e^g ; Q e^g]: 4 atoms x 128 rows x 128 B
constexpr uint32_t S1_OPB = 147456;   // tf32 K e^-g: 4 atoms x 64 rows x 128 B
constexpr uint32_t S1_KG16 = 180224;  // fp16 K e^g, [r][c] 128B-swizzled (MN-major B)
constexpr uint32_t S1_V16 = 196608;   // fp16 V, same layout
constexpr uint32_t S1_TP = 212992;    // fp16 T', K-major SW128 [r][i]
constexpr uint32_t S1_MISC = 221184;
constexpr uint32_t S1_BYTES = S1_MISC + 4096 + 1024;
// after the A/P MMA has completed the operand area is reused by the inverse:
constexpr int LD = 68;                          // fp32 row stride of the 64 x 64 tiles
constexpr uint32_t TILE_BYTES = 64 * LD * 4;    // 17,408
constexpr uint32_t S1_AS = S1_OPA;                   // A    fp32 [64][LD]
constexpr uint32_t S1_TS = S1_OPA + TILE_BYTES;      // T    fp32 [64][LD]
constexpr uint32_t S1_TT = S1_OPA + 2 * TILE_BYTES;  // T_RR transposed (diagonal blocks)
constexpr uint32_t S1_FT = S1_OPA + 3 * TILE_BYTES;  // F = T_RR A_RJ, transposed
static_assert(S1_FT + TILE_BYTES <= S1_KG16, "inverse scratch overlaps the fp16 operands");
constexpr int AP_COL = 0, W_COL = 256, U_COL = 384;  // TMEM: 4 A/P partials of 64, W, U~
constexpr float RANGE_LIMIT = 80.f;                   // e^80 stays inside fp32

struct K1Params {
    CUtensorMap tm_q, tm_k, tm_v, tm_g;   // 3D maps over [T][H][128] (tm_g unused for scalar gates)
    const float *g;                       // scalar gates [T][H] (when scalar_gate)
    const float *beta;
    const int32_t *cu;
    uint8_t *ws;
    int N, H;
    int64_t T;
    int w0, w1;
    int scalar_gate;
};

__device__ __forceinline__ void tma_load_3d(uint8_t *dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *mbar) {
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4}], [%5];"
                 :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1),
                    "r"(c2), "r"(smem_addr(mbar))
                 : "memory");
}

__device__ __forceinline__ uint4 pack8_h(const float *x) {
    return make_uint4(pack_h2(x[0], x[1]), pack_h2(x[2], x[3]), pack_h2(x[4], x[5]),
                      pack_h2(x[6], x[7]));
}

// [r][c] 128B-swizzled image with 64-channel atoms: byte offset of the 16-byte
// chunk holding channels c0..c0+7 of row r (c0 a multiple of 8).
__device__ __forceinline__ uint32_t rc_img_off(int r, int c0) {
    return (uint32_t)(c0 >> 6) * 8192u + sw128_off(r, (c0 & 63) >> 3);
}

// acc[2][4] += X[m0..m0+1][k] Y[k][n0..n0+3] over k = 0..15, with X read
// transposed (Xt[k][m]) and Y row-major, both with row stride LD.
__device__ __forceinline__ void mm16_2x4(float (&acc)[2][4], const float *Xt, const float *Y) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float2 x = *reinterpret_cast<const float2 *>(Xt + k * LD);
        const float4 y = *reinterpret_cast<const float4 *>(Y + k * LD);
        acc[0][0] = fmaf(x.x, y.x, acc[0][0]); acc[0][1] = fmaf(x.x, y.y, acc[0][1]);
        acc[0][2] = fmaf(x.x, y.z, acc[0][2]); acc[0][3] = fmaf(x.x, y.w, acc[0][3]);
        acc[1][0] = fmaf(x.y, y.x, acc[1][0]); acc[1][1] = fmaf(x.y, y.y, acc[1][1]);
        acc[1][2] = fmaf(x.y, y.z, acc[1][2]); acc[1][3] = fmaf(x.y, y.w, acc[1][3]);
    }
}

// fp16 of x at (row r, column i) of the K-major 128B-swizzled T' image
__device__ __forceinline__ void tp_store1(uint8_t *img, int r, int i, float x) {
    *reinterpret_cast<__half *>(img + sw128_off(r, i >> 3) + (i & 7) * 2) = __float2half_rn(x);
}

// T = (I + A)^-1 for the strictly lower 64 x 64 A (row-major, stride LD) in
// 16 x 16 blocks, fp32 on CUDA cores, and the fp16 image of T' = T Diag(beta).
// With T_RR the inverses of the diagonal blocks of I + A and F_RJ = T_RR A_RJ
// (J < R), block forward substitution gives T_RI = -sum_{J=I}^{R-1} F_RJ T_JI
// for I < R.  Six warps each own one off-diagonal block of T (2 x 4 outputs
// per lane, partial sums kept in registers) and add one term per pass, so the
// whole inverse is: diagonal blocks | F | three passes.  Run by warps 0-5
// only (named barrier 1), leaving the other warps free.  The image's blocks
// above the diagonal are not written (they hold zeros).
constexpr int INV_THREADS = 192;
__device__ __forceinline__ void invert_unit_lower(const float *As, float *Ts, float *Tt, float *Ft,
                                                  const float *sB, uint8_t *tp_img, int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    // diagonal blocks: thread (R, column j) by forward substitution in registers
    if (tid < 64) {
        const int R = tid >> 4, j = tid & 15;
        const float *Ab = As + (16 * R) * LD + 16 * R;
        float x[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) x[m] = (m == j) ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < 15; ++i) {
            const float xi = x[i];
#pragma unroll
            for (int r = i + 1; r < 16; ++r) x[r] = fmaf(-Ab[r * LD + i], xi, x[r]);
        }
        const float bj = sB[16 * R + j];
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            Ts[(16 * R + m) * LD + 16 * R + j] = x[m];
            tp_store1(tp_img, 16 * R + m, 16 * R + j, x[m] * bj);
        }
        float4 *trow = reinterpret_cast<float4 *>(Tt + (16 * R + j) * LD + 16 * R);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
            trow[q4] = make_float4(x[4 * q4], x[4 * q4 + 1], x[4 * q4 + 2], x[4 * q4 + 3]);
    }
    bar_sync(1, INV_THREADS);

    // warp w owns block (R, I): (1,0) (2,1) (3,2) (2,0) (3,1) (3,0)
    const int R = warp < 3 ? warp + 1 : (warp < 5 ? warp - 1 : 3);
    const int I = warp < 3 ? warp : (warp < 5 ? warp - 3 : 0);
    const int m0 = 2 * (lane >> 2), n0 = 4 * (lane & 3);
    {   // F_RI = T_RR A_RI, stored transposed
        float f[2][4] = {};
        mm16_2x4(f, Tt + (16 * R) * LD + 16 * R + m0, As + (16 * R) * LD + 16 * I + n0);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            *reinterpret_cast<float2 *>(Ft + (16 * I + n0 + e) * LD + 16 * R + m0) =
                make_float2(f[0][e], f[1][e]);
    }
    bar_sync(1, INV_THREADS);
    float acc[2][4] = {};
#pragma unroll
    for (int pass = 0; pass < 3; ++pass) {
        const int J = I + pass;
        if (J < R) {
            mm16_2x4(acc, Ft + (16 * J) * LD + 16 * R + m0, Ts + (16 * J) * LD + 16 * I + n0);
            if (J == R - 1) {
                const float4 b4 = *reinterpret_cast<const float4 *>(sB + 16 * I + n0);
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    const int r = 16 * R + m0 + a, i = 16 * I + n0;
                    *reinterpret_cast<float4 *>(Ts + r * LD + i) =
                        make_float4(-acc[a][0], -acc[a][1], -acc[a][2], -acc[a][3]);
                    *reinterpret_cast<uint2 *>(tp_img + sw128_off(r, i >> 3) + (i & 7) * 2) =
                        make_uint2(pack_h2(-acc[a][0] * b4.x, -acc[a][1] * b4.y),
                                   pack_h2(-acc[a][2] * b4.z, -acc[a][3] * b4.w));
                }
            }
        }
        if (pass < 2) bar_sync(1, INV_THREADS);
    }
}

__global__ void __launch_bounds__(K1_THREADS, 1) intra_kernel(const __grid_constant__ K1Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    float *gL = reinterpret_cast<float *>(sm + S1_MISC);   // [128] gamma_last
    float *eL = gL + 128;                                  // [128] e^gamma_last
    float *sB = eL + 128;                                  // [64] beta
    float *tot = sB + 64;                                  // [4][128] segment totals
    float *sGs = tot + 512;                                // [64] scalar gates (scalar_gate)
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sGs + 64);   // [0] TMA, [1] A/P, [2] W/U
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mbar + 3);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *ws_hdr = reinterpret_cast<int32_t *>(p.ws);
    const int32_t *chunk_base = reinterpret_cast<const int32_t *>(p.ws + WS_HEADER);
    uint8_t *img_base = p.ws + ws_images_offset(p.N);
    const int H = p.H;

    if (tid == 0) {
        mbar_init(&mbar[0], 1);
        mbar_init(&mbar[1], 4);   // four A/P issuers
        mbar_init(&mbar[2], 2);   // W and U~ issuers
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc<512>(tmem_slot);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // T' is lower triangular: the blocks above its diagonal stay zero (the
    // inverse rewrites only the diagonal and lower blocks)
    for (int e = tid; e < 64 * 8; e += K1_THREADS) {
        const int r = e >> 3, ch = e & 7;
        if (ch >= 2 * ((r >> 4) + 1))
            *reinterpret_cast<uint4 *>(sm + S1_TP + sw128_off(r, ch)) = make_uint4(0, 0, 0, 0);
    }

    const int total = chunk_base[p.N];
    const int c_end = min(p.w1, total);
    const int ntask = (c_end > p.w0 ? c_end - p.w0 : 0) * H;
    const int stride = gridDim.x;

    struct Pos { int h, L; int64_t t0; };
    // A task's position in two steps: fetch issues the offset-table loads,
    // finish is their first use (placed a phase later, so that the loads'
    // latency is hidden).  Together they give the sequence bounds clamped into
    // [0, T] (as seq_bounds does) and the chunk's first token and length.
    struct PosRaw { int ch, h; int32_t c0, c1, cb; };
    auto pos_fetch = [&](int task) {
        PosRaw r{-1, 0, 0, 0, 0};
        if (task >= ntask) return r;
        r.ch = p.w0 + task / H;
        r.h = task % H;
        const int n = find_seq(chunk_base, p.N, r.ch);
        r.c0 = p.cu[n];
        r.c1 = p.cu[n + 1];
        r.cb = chunk_base[n];
        return r;
    };
    auto pos_finish = [&](const PosRaw &r) {
        Pos q{0, 0, 0};
        if (r.ch < 0) return q;
        int64_t bos = r.c0, eos = r.c1;
        bos = bos < 0 ? 0 : (bos > p.T ? p.T : bos);
        eos = eos < bos ? bos : (eos > p.T ? p.T : eos);
        q.h = r.h;
        q.t0 = bos + (int64_t)(r.ch - r.cb) * C;
        q.L = (int)((eos - q.t0) < C ? (eos - q.t0) : C);
        return q;
    };
    auto task_pos = [&](int task) { return pos_finish(pos_fetch(task)); };
    // beta (and the scalar gate) of row `tid` of a task, read ahead into registers
    auto row_params = [&](const Pos &q, int task, float &b, float &gs) {
        b = 0.f; gs = 0.f;
        if (tid < C && task < ntask && tid < q.L) {
            b = p.beta[(q.t0 + tid) * H + q.h];
            if (p.scalar_gate) gs = p.g[(q.t0 + tid) * H + q.h];
        }
    };
    constexpr uint32_t TILE_BF16 = 16384, TILE_G = 32768;
    auto expect_tma = [&]() {
        mbar_arrive_expect_tx(&mbar[0], 3 * TILE_BF16 + (p.scalar_gate ? 0 : TILE_G));
    };
    auto tma_kqg = [&](const Pos &q) {
        tma_load_3d(sm + S1_STG_K, &p.tm_k, 0, q.h, (int)q.t0, &mbar[0]);
        tma_load_3d(sm + S1_STG_Q, &p.tm_q, 0, q.h, (int)q.t0, &mbar[0]);
        if (!p.scalar_gate) tma_load_3d(sm + S1_STG_G, &p.tm_g, 0, q.h, (int)q.t0, &mbar[0]);
    };
    auto tma_v = [&](const Pos &q) {
        tma_load_3d(sm + S1_STG_V, &p.tm_v, 0, q.h, (int)q.t0, &mbar[0]);
    };
    // W and U~ of a finished task: TMEM -> fp16 workspace images.  Row r of
    // the M = 64 accumulators sits in lane r % 16 of quadrant r / 16; a warp
    // reads its own quadrant.
    auto store_wu_cols = [&](uint8_t *dst, int q, int col) {   // 16 columns
        const int r = 16 * q + lane;
        float w[16], u[16];
        tmem_ld16(tmem_at(tmem, q, W_COL + col), w);
        tmem_ld16(tmem_at(tmem, q, U_COL + col), u);
        tmem_wait_ld();
        if (lane < 16) {
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                const int c0 = col + 8 * hc;
                *reinterpret_cast<uint4 *>(dst + IMG_W + rc_img_off(r, c0)) = pack8_h(w + 8 * hc);
                *reinterpret_cast<uint4 *>(dst + IMG_U + (c0 >> 5) * 4096 + r * 64 + (c0 & 31) * 2) =
                    pack8_h(u + 8 * hc);
            }
        }
    };
    auto store_wu = [&](uint8_t *dst) {        // all 16 warps: 32 columns each
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) store_wu_cols(dst, warp & 3, 32 * (warp >> 2) + 16 * hh);
    };
    // The same, split so that the TMEM loads' latency overlaps other work:
    // round hh (0, 1) of warp w covers columns 32 (w / 4) + 16 hh.
    auto drain_issue = [&](int hh, float (&w)[16], float (&u)[16]) {
        const int col = 32 * (warp >> 2) + 16 * hh;
        tmem_ld16(tmem_at(tmem, warp & 3, W_COL + col), w);
        tmem_ld16(tmem_at(tmem, warp & 3, U_COL + col), u);
    };
    auto drain_finish = [&](uint8_t *dst, int hh, float (&w)[16], float (&u)[16]) {
        tmem_wait_ld();
        reg_fence(w);
        reg_fence(u);
        const int col = 32 * (warp >> 2) + 16 * hh;
        const int r = 16 * (warp & 3) + lane;
        if (lane < 16) {
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                const int c0 = col + 8 * hc;
                *reinterpret_cast<uint4 *>(dst + IMG_W + rc_img_off(r, c0)) = pack8_h(w + 8 * hc);
                *reinterpret_cast<uint4 *>(dst + IMG_U + (c0 >> 5) * 4096 + r * 64 + (c0 & 31) * 2) =
                    pack8_h(u + 8 * hc);
            }
        }
    };

    // positions are resolved one task ahead of the one being loaded, so the
    // offset-table lookups never sit on the critical path
    int task = blockIdx.x;
    Pos cur = task_pos(task), nxt = task_pos(task + stride);
    float b_cur, gs_cur;
    row_params(cur, task, b_cur, gs_cur);
    uint32_t n_issued = 0, n_landed = 0;   // TMA phases (meaningful in thread 0, the issuer)
    if (tid == 0 && task < ntask) { expect_tma(); tma_kqg(cur); tma_v(cur); n_issued = 1; }

    bool ok = true;
    uint32_t it = 0, ap_it = 0;
    uint8_t *out_prev = nullptr;
    for (; task < ntask; task += stride, ++it) {
        const int L = cur.L;
        const int next = task + stride;
        uint8_t *out = img_base + (uint64_t)task * CH_STRIDE;
        if (tid < C) {
            sB[tid] = b_cur;
            sGs[tid] = gs_cur;
        }
        ok = __syncthreads_and(mbar_wait(&mbar[0], it & 1));
        if (!ok) break;
        ++n_landed;

        // ---- cumulative log-gate, in place (rows past the sequence: g = 0) ----
        // thread = (channel c, 16-row segment sg)
        {
            const int c = tid & 127, sg = tid >> 7;
            float *G = reinterpret_cast<float *>(sm + S1_STG_G);
            float v[16];
            if (p.scalar_gate) {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = sGs[16 * sg + j];
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = G[(16 * sg + j) * 128 + c];
            }
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                acc += 16 * sg + j < L ? v[j] : 0.f;
                v[j] = acc;
            }
            tot[sg * 128 + c] = acc;
            __syncthreads();
            float off = 0.f;
            for (int s2 = 0; s2 < sg; ++s2) off += tot[s2 * 128 + c];
#pragma unroll
            for (int j = 0; j < 16; ++j) G[(16 * sg + j) * 128 + c] = v[j] + off;
            if (sg == 3) {
                gL[c] = acc + off;
                eL[c] = __expf(acc + off);
            }
        }
        // The previous task's W/U MMA ran under the scan; it must be done before
        // the prep rewrites its B operands and before its results leave TMEM
        // (this task's W/U MMA reuses the columns), in two rounds hidden behind
        // the prep.
        ok = __syncthreads_and(it == 0 || mbar_wait(&mbar[2], (it - 1) & 1));
        fence_after_sync();
        if (!ok) break;
        const bool slow = __syncthreads_or(tid >= 384 && -gL[tid & 127] > RANGE_LIMIT);
        float dw[16], du[16];
        if (out_prev) drain_issue(0, dw, du);

        // ---- element-wise prep: unit = (row r, channels c0..c0+7) -------------
        // tf32 operands [K e^g ; Q e^g] and K e^-g for A / P (not on the slow
        // path), fp16 K e^g and V for W / U~, the Q^ and Kbar workspace images.
#pragma unroll 1
        for (int jj = 0; jj < 2; ++jj) {
            const int u = tid + K1_THREADS * jj;
            const int r = u >> 4, c0 = (u & 15) * 8;
            float kf[8], qf[8], vf[8], gm[8], el[8];
            {
                const uint4 kr = *reinterpret_cast<const uint4 *>(sm + S1_STG_K + r * 256 + c0 * 2);
                const uint4 qr = *reinterpret_cast<const uint4 *>(sm + S1_STG_Q + r * 256 + c0 * 2);
                const uint4 vr = *reinterpret_cast<const uint4 *>(sm + S1_STG_V + r * 256 + c0 * 2);
                const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&kr);
                const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&qr);
                const __nv_bfloat162 *v2 = reinterpret_cast<const __nv_bfloat162 *>(&vr);
                const bool live = r < L;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 a = __bfloat1622float2(k2[e]), b2 = __bfloat1622float2(q2[e]),
                                 c2 = __bfloat1622float2(v2[e]);
                    kf[2 * e] = live ? a.x : 0.f; kf[2 * e + 1] = live ? a.y : 0.f;
                    qf[2 * e] = live ? b2.x : 0.f; qf[2 * e + 1] = live ? b2.y : 0.f;
                    vf[2 * e] = live ? c2.x : 0.f; vf[2 * e + 1] = live ? c2.y : 0.f;
                }
                const float4 g0 = *reinterpret_cast<const float4 *>(sm + S1_STG_G + r * 512 + c0 * 4);
                const float4 g1 = *reinterpret_cast<const float4 *>(sm + S1_STG_G + r * 512 + c0 * 4 + 16);
                gm[0] = g0.x; gm[1] = g0.y; gm[2] = g0.z; gm[3] = g0.w;
                gm[4] = g1.x; gm[5] = g1.y; gm[6] = g1.z; gm[7] = g1.w;
                const float4 e0 = *reinterpret_cast<const float4 *>(eL + c0);
                const float4 e1 = *reinterpret_cast<const float4 *>(eL + c0 + 4);
                el[0] = e0.x; el[1] = e0.y; el[2] = e0.z; el[3] = e0.w;
                el[4] = e1.x; el[5] = e1.y; el[6] = e1.z; el[7] = e1.w;
            }
            float kg[8], qg[8], kh[8], kb[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float ep = __expf(gm[e]);
                kg[e] = kf[e] * ep;
                qg[e] = qf[e] * ep;
                if (!slow) {   // e^-gamma <= e^80 here: Kbar = (K e^-g) e^gamma_last
                    kh[e] = kf[e] * __expf(-gm[e]);
                    kb[e] = kh[e] * el[e];
                } else {
                    kh[e] = 0.f;
                    kb[e] = kf[e] * __expf(gL[c0 + e] - gm[e]);
                }
            }
            const uint32_t ioff = rc_img_off(r, c0);
            *reinterpret_cast<uint4 *>(sm + S1_KG16 + ioff) = pack8_h(kg);
            *reinterpret_cast<uint4 *>(sm + S1_V16 + ioff) = pack8_h(vf);
            *reinterpret_cast<uint4 *>(out + IMG_Q + ioff) = pack8_h(qg);
            *reinterpret_cast<uint4 *>(out + IMG_KT + ioff) = pack8_h(kb);
            if (!slow) {
                const uint32_t atom = (uint32_t)(c0 >> 5), ch0 = (uint32_t)(c0 & 31) >> 2;
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                    const uint32_t cc = ch0 + hc;
                    *reinterpret_cast<float4 *>(sm + S1_OPA + atom * 16384 + sw128_off(r, cc)) =
                        make_float4(kg[4 * hc], kg[4 * hc + 1], kg[4 * hc + 2], kg[4 * hc + 3]);
                    *reinterpret_cast<float4 *>(sm + S1_OPA + atom * 16384 + sw128_off(64 + r, cc)) =
                        make_float4(qg[4 * hc], qg[4 * hc + 1], qg[4 * hc + 2], qg[4 * hc + 3]);
                    *reinterpret_cast<float4 *>(sm + S1_OPB + atom * 8192 + sw128_off(r, cc)) =
                        make_float4(kh[4 * hc], kh[4 * hc + 1], kh[4 * hc + 2], kh[4 * hc + 3]);
                }
            }
            if (jj == 0 && out_prev) {
                drain_finish(out_prev, 0, dw, du);
                drain_issue(1, dw, du);
            }
        }
        if (out_prev) drain_finish(out_prev, 1, dw, du);
        if (tid < 128) reinterpret_cast<float *>(out + IMG_G)[tid] = eL[tid];
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ---- A and P: tf32 MMAs, M = 128 ([K e^g ; Q e^g]), N = 64 (K e^-g).
        // Issuing one keeps its thread busy for a few hundred cycles, so the
        // 16 K steps are spread over four issuers (warps 12-15, accumulator =
        // channel atom); warp 12 then starts the next task's loads (every
        // staging tile is consumed).  Meanwhile every thread resolves the
        // task after next.
        if (!slow && warp >= K1_ISSUER0 && lane == 0) {
            const int atom = warp - K1_ISSUER0;
            fence_after_sync();
            const uint64_t da = sdesc_k_sw128(smem_addr(sm + S1_OPA));
            const uint64_t db = sdesc_k_sw128(smem_addr(sm + S1_OPB));
            const uint32_t id = idesc(128, 64, FMT_TF32, FMT_TF32, 0, 0);
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) {   // 8 tf32 channels per step
                const uint32_t wi = s2 * 32;
                mma_tf32(tmem + AP_COL + 64 * atom, sdesc_add(da, atom * 16384 + wi),
                         sdesc_add(db, atom * 8192 + wi), id, s2 > 0);
            }
            mma_commit(&mbar[1]);
            if (atom == 0 && next < ntask) { expect_tma(); tma_kqg(nxt); tma_v(nxt); }
        }
        row_params(nxt, next, b_cur, gs_cur);              // consumed next task
        const PosRaw nn_raw = pos_fetch(next + stride);    // finished after the W/U MMA

        float *As = reinterpret_cast<float *>(sm + S1_AS);
        if (!slow) {
            if (tid == 0 && next < ntask) ++n_issued;
            fence_before_sync();
            ok = __syncthreads_and(mbar_wait(&mbar[1], ap_it & 1));
            ++ap_it;
            fence_after_sync();
            if (!ok) break;
            {   // warp = (lane quadrant q, 16-column block cb); lane = row
                const int q = warp & 3, cb = warp >> 2;
                const int row = 32 * q + lane;
                float d[16], d1[16], d2[16], d3[16];
                tmem_ld16(tmem_at(tmem, q, AP_COL + 16 * cb), d);
                tmem_ld16(tmem_at(tmem, q, AP_COL + 64 + 16 * cb), d1);
                tmem_ld16(tmem_at(tmem, q, AP_COL + 128 + 16 * cb), d2);
                tmem_ld16(tmem_at(tmem, q, AP_COL + 192 + 16 * cb), d3);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) d[e] = (d[e] + d1[e]) + (d2[e] + d3[e]);
                if (row < 64) {
                    const float b = sB[row];
                    float4 *arow = reinterpret_cast<float4 *>(As + row * LD + 16 * cb);
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                        float a4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = 16 * cb + 4 * e4 + e;
                            a4[e] = row > i ? b * d[4 * e4 + e] : 0.f;
                        }
                        arow[e4] = make_float4(a4[0], a4[1], a4[2], a4[3]);
                    }
                } else {
                    const int r = row - 64;
                    float pv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) pv[e] = (16 * cb + e) <= r ? d[e] : 0.f;
                    *reinterpret_cast<uint4 *>(out + IMG_P + sw128_off(r, 2 * cb)) = pack8_h(pv);
                    *reinterpret_cast<uint4 *>(out + IMG_P + sw128_off(r, 2 * cb + 1)) = pack8_h(pv + 8);
                }
            }
        } else {
            // ---- exact pairwise path for chunks whose decay leaves fp32 range
            const __nv_bfloat16 *Kb = reinterpret_cast<const __nv_bfloat16 *>(sm + S1_STG_K);
            const __nv_bfloat16 *Qb = reinterpret_cast<const __nv_bfloat16 *>(sm + S1_STG_Q);
            const float *Gm = reinterpret_cast<const float *>(sm + S1_STG_G);
            for (int e = tid; e < C * C; e += K1_THREADS) {
                const int r = e >> 6, i = e & 63;
                float a = 0.f, pp = 0.f;
                if (i <= r && r < L) {
                    for (int c = 0; c < D; ++c) {
                        const float ki = __bfloat162float(Kb[i * 128 + c]) *
                                         __expf(Gm[r * 128 + c] - Gm[i * 128 + c]);
                        a += __bfloat162float(Kb[r * 128 + c]) * ki;
                        pp += __bfloat162float(Qb[r * 128 + c]) * ki;
                    }
                }
                As[r * LD + i] = i < r ? sB[r] * a : 0.f;
                *reinterpret_cast<__half *>(out + IMG_P + sw128_off(r, i >> 3) + (i & 7) * 2) =
                    __float2half_rn(pp);
            }
            fence_before_sync();
            __syncthreads();
            if (tid == 0 && next < ntask) {   // staging is consumed
                expect_tma(); tma_kqg(nxt); tma_v(nxt);
                ++n_issued;
            }
        }
        __syncthreads();

        // ---- T = (I + A)^-1 and the fp16 image of T' = T Diag(beta) (warps 0-5)
        if (warp < 6)
            invert_unit_lower(As, reinterpret_cast<float *>(sm + S1_TS),
                              reinterpret_cast<float *>(sm + S1_TT),
                              reinterpret_cast<float *>(sm + S1_FT), sB, sm + S1_TP, tid);
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ---- W = T' (K e^g), U~ = T' V on tcgen05 (fp16, B operands MN-major);
        // warp 0 issues W, warp 1 issues U~
        if (lane == 0 && warp < 2) {
            fence_after_sync();
            const uint64_t dt = sdesc_k_sw128(smem_addr(sm + S1_TP));
            const uint64_t db = sdesc(smem_addr(sm + (warp == 0 ? S1_KG16 : S1_V16)), 8192, 1024,
                                      LAYOUT_SW128);
            const uint32_t id = idesc(64, 128, FMT_F16, FMT_F16, 0, 1);
            const uint32_t col = warp == 0 ? W_COL : U_COL;
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2)
                mma_f16(tmem + col, sdesc_add(dt, 32 * s2), sdesc_add(db, 2048 * s2), id, s2 > 0);
            mma_commit(&mbar[2]);   // waited for after the next task's gate scan
        }
        out_prev = out;
        cur = nxt;
        nxt = pos_finish(nn_raw);
    }
    // the last W/U MMA, then its results
    if (ok && it > 0) {
        ok = __syncthreads_and(mbar_wait(&mbar[2], (it - 1) & 1));
        fence_after_sync();
        if (ok) store_wu(out_prev);
    }
    if (!ok && tid == 0) {
        ws_fail(ws_hdr, 1);
        // let copies and MMAs still in flight finish before the CTA's shared
        // memory and TMEM are released (bounded waits)
        if (n_issued > n_landed) mbar_wait(&mbar[0], (n_issued - 1) & 1, 1u << 20);
        if (it > 0) mbar_wait(&mbar[2], (it - 1) & 1, 1u << 20);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc<512>(tmem);
}

// ------------------------------------------------------------------------------
// K2: chain kernel
// ------------------------------------------------------------------------------
// One CTA of 128 threads per (sequence, head, block of 32 state columns);
// thread t owns row t (a dk channel) of the fp32 state.  Per chunk:
//   round 1: D_A + D_B = [W ; Q^] S   (M = 128: rows 0-63 W S, 64-127 Q^ S;
//            K steps 0-3 into D_A by warp 0, 4-7 into D_B by warp 1)
//   U = U~ - W S (fp16);
//   round 2: D_S + D_S2 = Kbar^T U (warps 0 and 1, two K steps each),
//            D_A += [0 ; P] U (warp 2; rows 64-127 then hold O - Q^S_B)
//   S = Diag(e^gamma_last) S + D_S + D_S2.
// A thread issuing tcgen05.mma is busy for ~90 cycles per instruction, so the
// few MMAs on the state's critical path are spread over several issuing warps.
// TMEM accumulators alternate between two sets so that the outputs of chunk
// i are read while the MMAs of chunk i + 1 run.
constexpr int K2_THREADS = 128;
constexpr uint32_t S2_WQ = 0;          // [W ; Q^] K-major SW128, 2 atoms x 128 rows
constexpr uint32_t S2_KB = 32768;      // Kbar [r][c] SW128 (MN-major A)
constexpr uint32_t S2_PZ = 49152;      // [0 ; P] K-major SW128, 128 rows (rows 0-63 zero)
constexpr uint32_t S2_U = 65536;       // U~ slice [64][32] fp16
constexpr uint32_t S2_G = 69632;       // e^gamma_last [128] fp32
constexpr uint32_t S2_STAGE = 70656;   // bytes per stage (multiple of 1024)
constexpr uint32_t S2_SOP = 2 * S2_STAGE;                 // S fp16, K=128 x N=32, MN-major
constexpr uint32_t S2_UOP = S2_SOP + 8192;                // U fp16, K=64 x N=32, MN-major
constexpr uint32_t S2_MISC = S2_UOP + 4096;
constexpr uint32_t S2_BYTES = S2_MISC + 256 + 1024;
constexpr uint32_t S2_TX = 4 * 8192 + 16384 + 8192 + 4096 + 512;   // bytes landing per stage
// TMEM set s (0, 1) at column 128 s: D_A +0, D_B +32, D_S +64, D_S2 +96

struct K2Params {
    const float *S0;
    float *S_T;
    __nv_bfloat16 *o;
    const int32_t *cu;
    uint8_t *ws;
    int N, H;
    int64_t T;
    int w0, w1;
    // chunk-affine scan of one sequence (N = 1), see segment_launch_plan
    int nseg;          // 0: off; else the window's chunks in nseg segments
    int seg_len;       // chunks per segment
    int phase;         // 0: segment maps (and segment 0 itself), 1: segments 1..nseg-1
    float *smaps;      // [H][nseg][3][128][128] fp32: M_s, B_s, start state of segment s
};

// Roles of a chain CTA in a segment launch.
enum : int { SEG_FULL = 0, SEG_B = 1, SEG_M = 2 };
constexpr int SMAP_M = 0, SMAP_B = 1, SMAP_START = 2;
__host__ __device__ inline float *smap(float *smaps, int nseg, int h, int s, int which) {
    return smaps + ((((size_t)h * nseg + s) * 3 + which) << 14);   // 128 x 128 each
}

__global__ void __launch_bounds__(K2_THREADS, 1) chain_kernel(const K2Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + S2_MISC);   // [0..1] loads, [2] r1, [3] r2
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mbar + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const int unit = blockIdx.x;
    int slice = unit % NSLICE;
    int h = (unit / NSLICE) % H;
    int n = unit / (NSLICE * H);
    int32_t *ws_hdr = reinterpret_cast<int32_t *>(p.ws);
    const int32_t *chunk_base = reinterpret_cast<const int32_t *>(p.ws + WS_HEADER);
    const uint8_t *img_base = p.ws + ws_images_offset(p.N);

    // A segment launch (one sequence): phase 0 runs, per head, segment 0
    // itself (slices 0-3) and, for each later segment, its state
    // contribution from a zero start (B) and its homogeneous map from an
    // identity start with U~ = 0 (M), four slices each; phase 1 runs
    // segments 1.. from their start states.
    int role = SEG_FULL, seg = 0;
    if (p.nseg) {
        n = 0;
        if (p.phase == 0) {
            const int per_head = 4 + 8 * (p.nseg - 1);
            h = unit / per_head;
            const int r = unit % per_head;
            if (r < 4) {
                slice = r;
            } else {
                seg = 1 + (r - 4) / 8;
                role = ((r - 4) % 8) < 4 ? SEG_B : SEG_M;
                slice = (r - 4) % 4;
            }
        } else {
            const int per_head = 4 * (p.nseg - 1);
            h = unit / per_head;
            seg = 1 + (unit % per_head) / 4;
            slice = unit % 4;
        }
    }

    const int cb = chunk_base[n], ce = chunk_base[n + 1];
    int a = max(cb, p.w0), b = min(ce, p.w1);
    if (p.nseg) {
        const int sa = a + seg * p.seg_len;
        b = min(b, sa + p.seg_len);
        a = sa;
    }
    const int64_t sbase = ((int64_t)n * H + h) * D * D + (int64_t)tid * D + slice * DVS;
    if (cb == ce && !p.nseg) {            // empty sequence: pass the state through
        if (p.w0 == 0) {
            for (int j = 0; j < DVS; j += 4) {
                float4 x = p.S0 ? *reinterpret_cast<const float4 *>(p.S0 + sbase + j)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4 *>(p.S_T + sbase + j) = x;
            }
        }
        return;
    }
    // no chunk of this sequence in the window (a segment launch still runs an
    // empty segment: it maps its start state to itself)
    if (a >= b && !p.nseg) return;

    int64_t bos, eos;
    seq_bounds(p.cu, n, p.T, bos, eos);

    float S[DVS];
    if (role == SEG_M) {          // identity columns slice*32 .. slice*32+31
#pragma unroll
        for (int j = 0; j < DVS; ++j) S[j] = (tid == slice * DVS + j) ? 1.f : 0.f;
    } else if (role == SEG_B) {
#pragma unroll
        for (int j = 0; j < DVS; ++j) S[j] = 0.f;
    } else {
        const float *src = (a == cb) ? p.S0 : p.S_T;
        int64_t off = sbase;
        if (p.nseg && seg > 0) {  // the start state the combine step produced
            src = smap(p.smaps, p.nseg, h, seg, SMAP_START);
            off = (int64_t)tid * D + slice * DVS;
        }
#pragma unroll
        for (int j = 0; j < DVS; j += 4) {
            float4 x = src ? *reinterpret_cast<const float4 *>(src + off + j)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
        }
    }
    const bool write_o = role == SEG_FULL;
    const float u_scale = role == SEG_M ? 0.f : 1.f;   // the homogeneous map drops U~
    // the zero half of [0 ; P] in both stages
    for (int e = tid; e < 2 * 8192 / 16; e += K2_THREADS) {
        const int st = e / 512, off = (e % 512) * 16;
        *reinterpret_cast<uint4 *>(sm + st * S2_STAGE + S2_PZ + off) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (tid == 0) {
        mbar_init(&mbar[0], 1);
        mbar_init(&mbar[1], 1);
        mbar_init(&mbar[2], 2);   // round 1: two issuers
        mbar_init(&mbar[3], 3);   // round 2: three issuers
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc<256>(tmem_slot);
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    auto issue_loads = [&](int ch, int stage) {
        const uint8_t *src = img_base + ((uint64_t)(ch - p.w0) * H + h) * CH_STRIDE;
        uint8_t *dst = sm + stage * S2_STAGE;
        uint64_t *mb = &mbar[stage];
        mbar_arrive_expect_tx(mb, S2_TX);
        bulk_g2s(dst + S2_WQ, src + IMG_W, 8192, mb);              // W, k 0-63
        bulk_g2s(dst + S2_WQ + 8192, src + IMG_Q, 8192, mb);       // Q^, k 0-63
        bulk_g2s(dst + S2_WQ + 16384, src + IMG_W + 8192, 8192, mb);
        bulk_g2s(dst + S2_WQ + 24576, src + IMG_Q + 8192, 8192, mb);
        bulk_g2s(dst + S2_KB, src + IMG_KT, 16384, mb);
        bulk_g2s(dst + S2_PZ + 8192, src + IMG_P, 8192, mb);
        bulk_g2s(dst + S2_U, src + IMG_U + slice * 4096, 4096, mb);
        bulk_g2s(dst + S2_G, src + IMG_G, 512, mb);
    };
    if (tid == 0 && a < b) {
        issue_loads(a, 0);
        if (a + 1 < b) issue_loads(a + 1, 1);
    }

    const uint64_t d_sop = sdesc(smem_addr(sm + S2_SOP), 128, 2048, LAYOUT_NONE);
    const uint64_t d_uop = sdesc(smem_addr(sm + S2_UOP), 128, 1024, LAYOUT_NONE);
    const uint32_t id_wq = idesc(128, DVS, FMT_F16, FMT_F16, 0, 1);
    const uint32_t id_kb = idesc(128, DVS, FMT_F16, FMT_F16, 1, 1);

    // stores the O rows of a finished chunk (threads 64-127: row tid - 64)
    auto store_o = [&](int set, int64_t t0, int L) {
        if (warp >= 2) {
            float oa[16], ob[16], pa[16], pb[16];
            tmem_ld16(tmem_at(tmem, warp, 128 * set), oa);
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 16), ob);
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 32), pa);
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 48), pb);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) { oa[j] += pa[j]; ob[j] += pb[j]; }
            const int r = tid - 64;
            if (r < L) {
                __nv_bfloat16 *dst = p.o + ((t0 + r) * H + h) * D + slice * DVS;
#pragma unroll
                for (int gq = 0; gq < DVS / 8; ++gq) {
                    const float *src = gq < 2 ? oa + 8 * gq : ob + 8 * (gq - 2);
                    __nv_bfloat162 b0 = __floats2bfloat162_rn(src[0], src[1]);
                    __nv_bfloat162 b1 = __floats2bfloat162_rn(src[2], src[3]);
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(src[4], src[5]);
                    __nv_bfloat162 b3 = __floats2bfloat162_rn(src[6], src[7]);
                    *reinterpret_cast<uint4 *>(dst + 8 * gq) = make_uint4(
                        *reinterpret_cast<uint32_t *>(&b0), *reinterpret_cast<uint32_t *>(&b1),
                        *reinterpret_cast<uint32_t *>(&b2), *reinterpret_cast<uint32_t *>(&b3));
                }
            }
        }
    };

    bool ok = true;
    int64_t prev_t0 = 0;
    int prev_L = 0;
    for (int ch = a; ch < b; ++ch) {
        const int i = ch - a, stage = i & 1, set = i & 1;
        uint8_t *st = sm + stage * S2_STAGE;
        const uint32_t tset = tmem + 128 * set;
        const int64_t t0 = bos + (int64_t)(ch - cb) * C;
        const int L = (int)((eos - t0) < C ? (eos - t0) : C);
        ok = __syncthreads_and(mbar_wait(&mbar[stage], (i >> 1) & 1));
        if (!ok) break;

        // S (fp16) -> B operand [K = dk][N = 32], MN-major, no swizzle:
        // core matrix (8 K rows x 8 N) at (n/8) * 2048 + (k/8) * 128
#pragma unroll
        for (int gq = 0; gq < DVS / 8; ++gq) {
            uint4 v4 = make_uint4(pack_h2(S[8 * gq + 0], S[8 * gq + 1]), pack_h2(S[8 * gq + 2], S[8 * gq + 3]),
                                  pack_h2(S[8 * gq + 4], S[8 * gq + 5]), pack_h2(S[8 * gq + 6], S[8 * gq + 7]));
            *reinterpret_cast<uint4 *>(sm + S2_SOP + gq * 2048 + (tid >> 3) * 128 + (tid & 7) * 16) = v4;
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        if (lane == 0 && warp < 2) {      // round 1: warp w takes K atom w
            fence_after_sync();
            const uint64_t dwq = sdesc_k_sw128(smem_addr(st + S2_WQ));
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_f16(tset + 32 * warp, sdesc_add(dwq, warp * 16384 + s * 32),
                        sdesc_add(d_sop, 256 * (4 * warp + s)), id_wq, s > 0);
            mma_commit(&mbar[2]);
        }
        if (i > 0 && write_o) store_o(set ^ 1, prev_t0, prev_L);   // previous chunk's outputs
        ok = __syncthreads_and(mbar_wait(&mbar[2], i & 1));
        fence_after_sync();
        if (!ok) break;

        // U = U~ - W S for token rows 0-63 (threads 0-63)
        if (warp < 2) {
            float w0[16], w1[16], x0[16], x1[16];
            tmem_ld16(tmem_at(tmem, warp, 128 * set), w0);
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 16), w1);
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 32), x0);
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 48), x1);
            tmem_wait_ld();
            const int r = tid;
            const __half *ut = reinterpret_cast<const __half *>(st + S2_U) + r * DVS;
            float u[DVS];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                u[j] = u_scale * __half2float(ut[j]) - (w0[j] + x0[j]);
                u[16 + j] = u_scale * __half2float(ut[16 + j]) - (w1[j] + x1[j]);
            }
#pragma unroll
            for (int gq = 0; gq < DVS / 8; ++gq) {
                uint4 v4 = make_uint4(pack_h2(u[8 * gq + 0], u[8 * gq + 1]), pack_h2(u[8 * gq + 2], u[8 * gq + 3]),
                                      pack_h2(u[8 * gq + 4], u[8 * gq + 5]), pack_h2(u[8 * gq + 6], u[8 * gq + 7]));
                *reinterpret_cast<uint4 *>(sm + S2_UOP + gq * 1024 + (r >> 3) * 128 + (r & 7) * 16) = v4;
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        if (lane == 0 && warp < 3) {      // round 2: warps 0-1 Kbar^T U halves, warp 2 P U
            fence_after_sync();
            if (warp < 2) {
                const uint64_t dkb = sdesc(smem_addr(st + S2_KB), 8192, 1024, LAYOUT_SW128);
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    const int ks = 2 * warp + s;
                    mma_f16(tset + 64 + 32 * warp, sdesc_add(dkb, 2048 * ks),
                            sdesc_add(d_uop, 256 * ks), id_kb, s > 0);
                }
            } else {
                const uint64_t dpz = sdesc_k_sw128(smem_addr(st + S2_PZ));
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16(tset, sdesc_add(dpz, 32 * s), sdesc_add(d_uop, 256 * s), id_wq, 1);
            }
            mma_commit(&mbar[3]);
        }
        ok = __syncthreads_and(mbar_wait(&mbar[3], i & 1));
        fence_after_sync();
        if (!ok) break;

        // S = Diag(e^gamma_last) S + Kbar^T U
        {
            float d2a[16], d2b[16], d3a[16], d3b[16];
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 64), d2a);
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 80), d2b);
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 96), d3a);
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 112), d3b);
            tmem_wait_ld();
            const float gl = reinterpret_cast<const float *>(st + S2_G)[tid];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                S[j] = gl * S[j] + (d2a[j] + d3a[j]);
                S[16 + j] = gl * S[16 + j] + (d2b[j] + d3b[j]);
            }
        }
        prev_t0 = t0;
        prev_L = L;
        fence_before_sync();
        __syncthreads();   // every thread is done with this stage
        if (tid == 0 && ch + 2 < b) issue_loads(ch + 2, stage);
    }
    if (ok && write_o && a < b) store_o((b - 1 - a) & 1, prev_t0, prev_L);

    if (!ok && tid == 0) ws_fail(ws_hdr, 2);
    // final state: S_T, or (segment launch) the segment's map, contribution
    // or end state for the combine step; the last segment writes S_T
    float *dst = nullptr;
    if (!p.nseg || (p.phase == 1 && seg == p.nseg - 1))
        dst = p.S_T + sbase;
    else if (p.phase == 0)   // segment 0 ends in its B slot
        dst = smap(p.smaps, p.nseg, h, seg, role == SEG_M ? SMAP_M : SMAP_B) + (int64_t)tid * D +
              slice * DVS;
    if (dst) {
#pragma unroll
        for (int j = 0; j < DVS; j += 4)
            *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc<256>(tmem);
}

// Chunk-affine scan, combine step: a segment maps its start state S to
// M_s S + B_s, so the start states follow in order from segment 0's end
// state (stored in its B slot).  One CTA per (head, 32-column slice), fp32 on
// CUDA cores: thread (row t, group of 8 columns); M_s is staged transposed in
// shared memory (rows padded to 129 floats) so that a warp reads consecutive
// rows of one column, and the slice of S is broadcast from shared memory
// (rows of 40 floats, so that a thread's 8 columns are two 16-byte loads).
constexpr int COMB_THREADS = 512;
constexpr int SSH_LD = 40;
constexpr uint32_t COMB_BYTES = (128 * 129 + 128 * SSH_LD) * sizeof(float);
__global__ void __launch_bounds__(COMB_THREADS) segment_combine_kernel(float *smaps, int nseg) {
    extern __shared__ float csm[];
    float *Mt = csm;                  // [k][t] = M_s[t][k], row stride 129
    float *Ssh = csm + 128 * 129;     // [k][j], row stride SSH_LD (16-byte aligned rows)
    const int h = blockIdx.x / NSLICE, slice = blockIdx.x % NSLICE;
    const int tid = threadIdx.x, t = tid & 127, g = tid >> 7;
    const int64_t off = (int64_t)t * D + slice * DVS + 8 * g;
    float S[8];
    const float *e0 = smap(smaps, nseg, h, 0, SMAP_B) + off;
#pragma unroll
    for (int j = 0; j < 8; ++j) S[j] = e0[j];
    for (int sg = 1; sg < nseg; ++sg) {
        float *start = smap(smaps, nseg, h, sg, SMAP_START) + off;
#pragma unroll
        for (int j = 0; j < 8; ++j) start[j] = S[j];
        if (sg == nseg - 1) break;
        __syncthreads();   // the previous step is done with Mt and Ssh
        const float4 *M4 = reinterpret_cast<const float4 *>(smap(smaps, nseg, h, sg, SMAP_M));
        for (int e = tid; e < 128 * 32; e += COMB_THREADS) {
            const int row = e >> 5, k4 = (e & 31) * 4;
            const float4 m = M4[e];
            Mt[(k4 + 0) * 129 + row] = m.x;
            Mt[(k4 + 1) * 129 + row] = m.y;
            Mt[(k4 + 2) * 129 + row] = m.z;
            Mt[(k4 + 3) * 129 + row] = m.w;
        }
        *reinterpret_cast<float4 *>(Ssh + t * SSH_LD + 8 * g) = make_float4(S[0], S[1], S[2], S[3]);
        *reinterpret_cast<float4 *>(Ssh + t * SSH_LD + 8 * g + 4) = make_float4(S[4], S[5], S[6], S[7]);
        __syncthreads();
        const float *Bv = smap(smaps, nseg, h, sg, SMAP_B) + off;
#pragma unroll
        for (int j = 0; j < 8; ++j) S[j] = Bv[j];
#pragma unroll 4
        for (int k = 0; k < D; ++k) {
            const float m = Mt[k * 129 + t];
            const float4 s0 = *reinterpret_cast<const float4 *>(Ssh + k * SSH_LD + 8 * g);
            const float4 s1 = *reinterpret_cast<const float4 *>(Ssh + k * SSH_LD + 8 * g + 4);
            S[0] = fmaf(m, s0.x, S[0]); S[1] = fmaf(m, s0.y, S[1]);
            S[2] = fmaf(m, s0.z, S[2]); S[3] = fmaf(m, s0.w, S[3]);
            S[4] = fmaf(m, s1.x, S[4]); S[5] = fmaf(m, s1.y, S[5]);
            S[6] = fmaf(m, s1.z, S[6]); S[7] = fmaf(m, s1.w, S[7]);
        }
    }
}

// ------------------------------------------------------------------------------
// K2, wide form: one CTA of 512 threads per (sequence, head), for batches
// with more chains than the GPU runs at once.  Warpgroup s (warps 4s..4s+3)
// owns state columns 32s..32s+31; its thread t (0..127) holds row t (a dk
// channel) of those columns in fp32 registers.  Every MMA spans the whole
// state (N = 128), so one SM carries a whole head.  Per chunk:
//   round 1: A_s + B_s = [W ; Q^] S   (M = 128, K = dk, split in halves over
//            two issuers; rows 0-63 W S, 64-127 Q^ S)
//   U = U~ - W S (fp16)                (rows 0-63: warps 0-1 of every warpgroup)
//   round 2: B_s' = Kbar^T U           (M = 128, K = 64; first issuer)
//            A_s += [0 ; P] U          (second issuer; rows 64-127 of A_s + B_s
//                                       then hold O)
//   S = Diag(e^gamma_last) S + B_s'.
// TMEM holds two 128-column accumulators per set; chunk c uses set s = c % 2
// for round 1 and the other set's B (whose previous contents, the last
// chunk's outputs, have left TMEM during round 1) for Kbar^T U.  Operand
// images arrive with bulk async copies, double buffered; a stage is reloaded
// once the next chunk's round 1 is issued, when its last reader (the P U MMA)
// has long finished.
constexpr int K2W_THREADS = 512;
constexpr uint32_t S2W_WQ = 0;          // [W ; Q^] K-major SW128, 2 atoms x 128 rows
constexpr uint32_t S2W_KB = 32768;      // Kbar [r][c] SW128 (MN-major A)
constexpr uint32_t S2W_PZ = 49152;      // [0 ; P] K-major SW128, 128 rows (rows 0-63 zero)
constexpr uint32_t S2W_U = 65536;       // U~ [4 column blocks][64][32] fp16
constexpr uint32_t S2W_G = 81920;       // e^gamma_last [128] fp32
constexpr uint32_t S2W_STAGE = 82944;   // bytes per stage (multiple of 1024)
constexpr uint32_t S2W_SOP = 2 * S2W_STAGE;                 // S fp16, K = 128 x N = 128, MN-major
constexpr uint32_t S2W_UOP = S2W_SOP + 32768;               // U fp16, K = 64 x N = 128, MN-major
constexpr uint32_t S2W_MISC = S2W_UOP + 16384;
constexpr uint32_t S2W_BYTES = S2W_MISC + 256 + 1024;
constexpr uint32_t S2W_TX = 4 * 8192 + 16384 + 8192 + 16384 + 512;   // bytes landing per stage
// TMEM set s (0, 1) at column 256 s: A_s +0, B_s +128

__global__ void __launch_bounds__(K2W_THREADS, 1) chain_wide_kernel(const K2Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    // [0..1] loads, [2] round 1 (two issuers), [3] round 2 state, [4] round 2 outputs
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + S2W_MISC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mbar + 5);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wg = warp >> 2, wq = warp & 3;   // column block, TMEM lane quadrant
    const int row = 32 * wq + lane;            // state row (dk channel) / TMEM lane
    const int col0 = 32 * wg;                  // first state column of this thread
    const int H = p.H;
    const int h = blockIdx.x % H;
    const int n = blockIdx.x / H;
    int32_t *ws_hdr = reinterpret_cast<int32_t *>(p.ws);
    const int32_t *chunk_base = reinterpret_cast<const int32_t *>(p.ws + WS_HEADER);
    const uint8_t *img_base = p.ws + ws_images_offset(p.N);

    const int cb = chunk_base[n], ce = chunk_base[n + 1];
    const int a = max(cb, p.w0), b = min(ce, p.w1);
    const int64_t sbase = ((int64_t)n * H + h) * D * D + (int64_t)row * D + col0;
    if (cb == ce) {                       // empty sequence: pass the state through
        if (p.w0 == 0) {
            for (int j = 0; j < 32; j += 4) {
                float4 x = p.S0 ? *reinterpret_cast<const float4 *>(p.S0 + sbase + j)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4 *>(p.S_T + sbase + j) = x;
            }
        }
        return;
    }
    if (a >= b) return;                   // no chunk of this sequence in the window

    int64_t bos, eos;
    seq_bounds(p.cu, n, p.T, bos, eos);

    float S[32];
    {
        const float *src = (a == cb) ? p.S0 : p.S_T;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            float4 x = src ? *reinterpret_cast<const float4 *>(src + sbase + j)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
        }
    }
    // the zero half of [0 ; P] in both stages
    for (int e = tid; e < 2 * 8192 / 16; e += K2W_THREADS) {
        const int st = e / 512, off = (e % 512) * 16;
        *reinterpret_cast<uint4 *>(sm + st * S2W_STAGE + S2W_PZ + off) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (tid == 0) {
        for (int j = 0; j < 5; ++j) mbar_init(&mbar[j], j == 2 ? 2 : 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc<512>(tmem_slot);
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    auto issue_loads = [&](int ch, int stage) {
        const uint8_t *src = img_base + ((uint64_t)(ch - p.w0) * H + h) * CH_STRIDE;
        uint8_t *dst = sm + stage * S2W_STAGE;
        uint64_t *mb = &mbar[stage];
        mbar_arrive_expect_tx(mb, S2W_TX);
        bulk_g2s(dst + S2W_WQ, src + IMG_W, 8192, mb);              // W, k 0-63
        bulk_g2s(dst + S2W_WQ + 8192, src + IMG_Q, 8192, mb);       // Q^, k 0-63
        bulk_g2s(dst + S2W_WQ + 16384, src + IMG_W + 8192, 8192, mb);
        bulk_g2s(dst + S2W_WQ + 24576, src + IMG_Q + 8192, 8192, mb);
        bulk_g2s(dst + S2W_KB, src + IMG_KT, 16384, mb);
        bulk_g2s(dst + S2W_PZ + 8192, src + IMG_P, 8192, mb);
        bulk_g2s(dst + S2W_U, src + IMG_U, 16384, mb);
        bulk_g2s(dst + S2W_G, src + IMG_G, 512, mb);
    };
    if (tid == 0) {
        issue_loads(a, 0);
        if (a + 1 < b) issue_loads(a + 1, 1);
    }
    // chunk a + 1 is loaded up front; chunk c + 1 for c > a is loaded during
    // chunk c (see round 1)

    const uint64_t d_sop = sdesc(smem_addr(sm + S2W_SOP), 128, 2048, LAYOUT_NONE);
    const uint64_t d_uop = sdesc(smem_addr(sm + S2W_UOP), 128, 1024, LAYOUT_NONE);
    const uint32_t id_wq = idesc(128, 128, FMT_F16, FMT_F16, 0, 1);
    const uint32_t id_kb = idesc(128, 128, FMT_F16, FMT_F16, 1, 1);

    // O rows of a finished chunk (TMEM lanes 64-127: warps 2-3 of each group)
    auto store_o = [&](int set, uint32_t phase, int64_t t0, int L) {
        if (wq >= 2) {
            const bool done = mbar_wait(&mbar[4], phase & 1);
            fence_after_sync();
            float oa[16], ob[16], pa[16], pb[16];
            tmem_ld16(tmem_at(tmem, wq, 256 * set + col0), oa);
            tmem_ld16(tmem_at(tmem, wq, 256 * set + col0 + 16), ob);
            tmem_ld16(tmem_at(tmem, wq, 256 * set + 128 + col0), pa);
            tmem_ld16(tmem_at(tmem, wq, 256 * set + 128 + col0 + 16), pb);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) { oa[j] += pa[j]; ob[j] += pb[j]; }
            const int r = row - 64;
            if (done && r < L) {
                __nv_bfloat16 *dst = p.o + ((t0 + r) * H + h) * D + col0;
#pragma unroll
                for (int gq = 0; gq < 4; ++gq) {
                    const float *src = gq < 2 ? oa + 8 * gq : ob + 8 * (gq - 2);
                    __nv_bfloat162 b0 = __floats2bfloat162_rn(src[0], src[1]);
                    __nv_bfloat162 b1 = __floats2bfloat162_rn(src[2], src[3]);
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(src[4], src[5]);
                    __nv_bfloat162 b3 = __floats2bfloat162_rn(src[6], src[7]);
                    *reinterpret_cast<uint4 *>(dst + 8 * gq) = make_uint4(
                        *reinterpret_cast<uint32_t *>(&b0), *reinterpret_cast<uint32_t *>(&b1),
                        *reinterpret_cast<uint32_t *>(&b2), *reinterpret_cast<uint32_t *>(&b3));
                }
            }
            return done;
        }
        return true;
    };

    bool ok = true;
    int64_t prev_t0 = 0;
    int prev_L = 0;
    for (int ch = a; ch < b; ++ch) {
        const int i = ch - a, stage = i & 1, set = i & 1;
        uint8_t *st = sm + stage * S2W_STAGE;
        const uint32_t acc_a = tmem + 256 * set, acc_b = acc_a + 128;   // round 1
        const uint32_t acc_s = tmem + 256 * (set ^ 1) + 128;              // Kbar^T U
        const int64_t t0 = bos + (int64_t)(ch - cb) * C;
        const int L = (int)((eos - t0) < C ? (eos - t0) : C);
        ok = __syncthreads_and(mbar_wait(&mbar[stage], (i >> 1) & 1));
        if (!ok) break;

        // S (fp16) -> B operand [K = dk][N = 128], MN-major, no swizzle:
        // core matrix (8 K rows x 8 N) at (n/8) * 2048 + (k/8) * 128
#pragma unroll
        for (int gq = 0; gq < 4; ++gq) {
            uint4 v4 = make_uint4(pack_h2(S[8 * gq + 0], S[8 * gq + 1]), pack_h2(S[8 * gq + 2], S[8 * gq + 3]),
                                  pack_h2(S[8 * gq + 4], S[8 * gq + 5]), pack_h2(S[8 * gq + 6], S[8 * gq + 7]));
            *reinterpret_cast<uint4 *>(sm + S2W_SOP + (4 * wg + gq) * 2048 + (row >> 3) * 128 + (row & 7) * 16) = v4;
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        if (lane == 0 && warp < 2) {      // round 1: warp w takes K atom w
            fence_after_sync();
            const uint64_t dwq = sdesc_k_sw128(smem_addr(st + S2W_WQ));
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4)
                mma_f16(warp == 0 ? acc_a : acc_b, sdesc_add(dwq, warp * 16384 + s4 * 32),
                        sdesc_add(d_sop, 256 * (4 * warp + s4)), id_wq, s4 > 0);
            mma_commit(&mbar[2]);
            // the previous chunk's P U MMA was the last reader of the other
            // stage: reload it with the chunk after next
            if (warp == 0 && i > 0 && ch + 1 < b) {
                if (mbar_wait(&mbar[4], (i - 1) & 1)) issue_loads(ch + 1, stage ^ 1);
                else ws_fail(ws_hdr, 2);
            }
        }
        bool o_ok = true;
        if (i > 0) o_ok = store_o(set ^ 1, (uint32_t)(i - 1), prev_t0, prev_L);
        ok = __syncthreads_and(mbar_wait(&mbar[2], i & 1) && o_ok);
        fence_after_sync();
        if (!ok) break;

        // U = U~ - W S for token rows 0-63 (warps 0-1 of each group)
        if (wq < 2) {
            float w0[16], w1[16], x0[16], x1[16];
            tmem_ld16(tmem_at(tmem, wq, 256 * set + col0), w0);
            tmem_ld16(tmem_at(tmem, wq, 256 * set + col0 + 16), w1);
            tmem_ld16(tmem_at(tmem, wq, 256 * set + 128 + col0), x0);
            tmem_ld16(tmem_at(tmem, wq, 256 * set + 128 + col0 + 16), x1);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) { w0[j] += x0[j]; w1[j] += x1[j]; }
            const int r = row;
            const uint4 *ut = reinterpret_cast<const uint4 *>(st + S2W_U + wg * 4096 + r * 64);
            float u[32];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const uint4 x = ut[q4];
                const __half2 *h2 = reinterpret_cast<const __half2 *>(&x);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(h2[e]);
                    const int j = 8 * q4 + 2 * e;
                    const float wa = j < 16 ? w0[j] : w1[j - 16];
                    const float wb = j + 1 < 16 ? w0[j + 1] : w1[j - 15];
                    u[j] = f.x - wa;
                    u[j + 1] = f.y - wb;
                }
            }
#pragma unroll
            for (int gq = 0; gq < 4; ++gq) {
                uint4 v4 = make_uint4(pack_h2(u[8 * gq + 0], u[8 * gq + 1]), pack_h2(u[8 * gq + 2], u[8 * gq + 3]),
                                      pack_h2(u[8 * gq + 4], u[8 * gq + 5]), pack_h2(u[8 * gq + 6], u[8 * gq + 7]));
                *reinterpret_cast<uint4 *>(sm + S2W_UOP + (4 * wg + gq) * 1024 + (r >> 3) * 128 + (r & 7) * 16) = v4;
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        if (lane == 0 && warp < 2) {      // round 2: warp 0 Kbar^T U, warp 1 [0 ; P] U
            fence_after_sync();
            if (warp == 0) {
                const uint64_t dkb = sdesc(smem_addr(st + S2W_KB), 8192, 1024, LAYOUT_SW128);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16(acc_s, sdesc_add(dkb, 2048 * ks), sdesc_add(d_uop, 256 * ks), id_kb, ks > 0);
                mma_commit(&mbar[3]);
            } else {
                const uint64_t dpz = sdesc_k_sw128(smem_addr(st + S2W_PZ));
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16(acc_a, sdesc_add(dpz, 32 * ks), sdesc_add(d_uop, 256 * ks), id_wq, 1);
                mma_commit(&mbar[4]);
            }
        }
        ok = __syncthreads_and(mbar_wait(&mbar[3], i & 1));
        fence_after_sync();
        if (!ok) break;

        // S = Diag(e^gamma_last) S + Kbar^T U
        {
            float da[16], db[16];
            tmem_ld16(tmem_at(tmem, wq, 256 * (set ^ 1) + 128 + col0), da);
            tmem_ld16(tmem_at(tmem, wq, 256 * (set ^ 1) + 128 + col0 + 16), db);
            tmem_wait_ld();
            const float gl = reinterpret_cast<const float *>(st + S2W_G)[row];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                S[j] = gl * S[j] + da[j];
                S[16 + j] = gl * S[16 + j] + db[j];
            }
        }
        prev_t0 = t0;
        prev_L = L;
        fence_before_sync();
        __syncthreads();   // every thread is done with this stage's images
    }
    if (ok) ok = __syncthreads_and(store_o((b - 1 - a) & 1, (uint32_t)(b - 1 - a), prev_t0, prev_L));

    if (!ok && tid == 0) ws_fail(ws_hdr, 2);
#pragma unroll
    for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4 *>(p.S_T + sbase + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc<512>(tmem);
}

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

// 3D map over a token-major [T][H][128] tensor; one box = 64 tokens of one head.
bool token_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, uint32_t esize, int H,
               int64_t T) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)H * D * esize};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)C};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int cached = 0;
    if (!cached) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&cached, cudaDevAttrMultiProcessorCount, dev);
        if (cached <= 0) cached = 1;
    }
    return cached;
}

}  // namespace

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
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)S1_BYTES);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S2_BYTES);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chain_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)S2W_BYTES);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(segment_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)COMB_BYTES);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    float *smaps = nullptr;
    if (scan) {
        const size_t images = (size_t)ws_images_offset(a.N) + (size_t)window * (size_t)a.H * CH_STRIDE;
        smaps = reinterpret_cast<float *>(ws + ((images + 255) & ~(size_t)255));
    }
    int32_t *hdr = reinterpret_cast<int32_t *>(ws);
    const int64_t bound = (a.T + C - 1) / C + a.N;
    chunk_table_kernel<<<1, 1024, 0, st>>>(a.cu_seqlens, a.N, a.T, (int)bound, hdr,
                                          reinterpret_cast<int32_t *>(ws + WS_HEADER));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int nsm = sm_count();
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
    p1.beta = a.beta; p1.cu = a.cu_seqlens; p1.ws = ws; p1.N = a.N; p1.H = a.H; p1.T = a.T;
    for (int64_t w0 = 0; w0 < bound; w0 += window) {
        const int64_t w1 = w0 + window;
        p1.w0 = (int)w0; p1.w1 = (int)w1;
        if (a.T > 0) {
            const int64_t tasks = (w1 - w0) * a.H;
            const int g1 = (int)(tasks < nsm ? tasks : nsm);
            intra_kernel<<<g1, K1_THREADS, S1_BYTES, st>>>(p1);
            e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        K2Params p2;
        p2.S0 = a.S0; p2.S_T = a.S_T; p2.o = (__nv_bfloat16 *)a.o; p2.cu = a.cu_seqlens;
        p2.ws = ws; p2.N = a.N; p2.H = a.H; p2.T = a.T; p2.w0 = (int)w0; p2.w1 = (int)w1;
        p2.nseg = 0; p2.seg_len = 0; p2.phase = 0; p2.smaps = smaps;
        const int64_t wch = (bound - w0) < window ? (bound - w0) : window;
        const SegPlan pl = smaps ? segment_plan(a.N, a.H, wch) : SegPlan{0, 0};
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
        // slices gets through about twice the chains per SM.
        const int64_t slices = (int64_t)a.N * a.H * NSLICE;
        if (slices > 2 * (int64_t)nsm)
            chain_wide_kernel<<<(unsigned)((int64_t)a.N * a.H), K2W_THREADS, S2W_BYTES, st>>>(p2);
        else
            chain_kernel<<<(unsigned)slices, K2_THREADS, S2_BYTES, st>>>(p2);
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

cudaError_t launch_prefill_tc_noalloc(const PrefillArgs &a, cudaStream_t st) {
    // device address of the scratch array, looked up once per device with
    // that device current (host code cannot use the symbol itself)
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    void *ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!addr[dev]) {
            e = cudaGetSymbolAddress(&addr[dev], g_noalloc_scratch);
            if (e != cudaSuccess) {
                addr[dev] = nullptr;
                return e;
            }
        }
        ws = addr[dev];
    }
    const int64_t window = noalloc_window_chunks(a.N, a.H);
    if (window < 1) return cudaErrorInvalidValue;
    return run_prefill_tc(a, static_cast<uint8_t *>(ws), window, false, st);
}

}  // namespace kda
