// kda_prefill_tc.cuh -- chunked KDA prefill on the 5th-generation tensor cores
// (tcgen05 + TMEM), bf16 inputs, fp32 state: the workspace and shared-memory
// layouts, kernel parameters and kernel declarations shared by
// kda_prefill_intra.cu (the per-chunk kernel), kda_prefill_chain.cu (the state
// chain) and kda_prefill_tc.cu (the host side).
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
#pragma once

#include "kda_internal.cuh"
#include "kda_tc.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

namespace kda {
namespace tcp {

using namespace tc;

constexpr int C = 64;          // tokens per chunk
constexpr int D = 128;         // dk = dv
constexpr int DVS = 32;        // state columns per chain CTA
constexpr int NSLICE = D / DVS;

// workspace: header | chunk table | chain plan | per (chunk, head) operand images
constexpr uint32_t WS_HEADER = 256;
constexpr uint32_t IMG_W = 0;          // W   [64 x 128] fp16, K-major SW128 (2 atoms)
constexpr uint32_t IMG_Q = 16384;      // Q^  [64 x 128] fp16, K-major SW128 (2 atoms)
constexpr uint32_t IMG_KT = 32768;     // Kb [64 x 128] fp16, [r][c] SW128 (MN-major A)
constexpr uint32_t IMG_P = 49152;      // P   [64 x 64] fp16, K-major SW128
constexpr uint32_t IMG_U = 57344;      // U~  [4 slices][64][32] fp16 (u_img_off)
constexpr uint32_t IMG_G = 73728;      // e^gamma_last [128] fp32
constexpr uint32_t CH_STRIDE = 74240;  // bytes per (chunk, head)
constexpr int WINDOW_CHUNKS = 2048;    // chunks per K1/K2 window

// Chain plan of a window (batches of many sequences): [0] the chain form
// (PLAN_SLICE or PLAN_WIDE), [1] the number of sequences listed, [2 ..] those
// sequences, longest chain in the window first.
constexpr int PLAN_SLICE = 0, PLAN_WIDE = 1;
__host__ __device__ inline uint64_t ws_plan_offset(int N) {
    return WS_HEADER + 4ull * (uint64_t)(N + 1);
}
__host__ __device__ inline uint64_t ws_images_offset(int N) {
    uint64_t off = ws_plan_offset(N) + 4ull * (uint64_t)(N + 2);
    return (off + 1023) & ~1023ull;
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

// U~ image of one 32-column state slice, [64 rows][32] fp16 (64 bytes a row):
// byte offset of the 16-byte chunk q (columns 8q..8q+7) of row r.  The chunk
// index is XOR-ed with bits 1-2 of the row, so that the 16-byte loads of 32
// consecutive rows (one per lane) hit distinct bank groups.
__host__ __device__ __forceinline__ uint32_t u_img_off(int r, int q) {
    return (uint32_t)r * 64u + ((uint32_t)(q ^ ((r >> 1) & 3)) << 4);
}

// byte offsets in the staging tiles: token t, channel c of a bf16 tile (boxes
// of 64 channels) and of an fp32 tile (boxes of 32 channels)
__host__ __device__ __forceinline__ uint32_t stg16_off(int t, int c) {
    return (uint32_t)(c >> 6) * 8192u + sw128_off((uint32_t)t, (uint32_t)(c & 63) >> 3) +
           (uint32_t)(c & 7) * 2u;
}
__host__ __device__ __forceinline__ uint32_t stg32_off(int t, int c) {
    return (uint32_t)(c >> 5) * 8192u + sw128_off((uint32_t)t, (uint32_t)(c & 31) >> 2) +
           (uint32_t)(c & 3) * 4u;
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// ---- per-chunk kernel: shared-memory layout and parameters ------------------
constexpr int K1_THREADS = 512;
constexpr int K1_ISSUER0 = 12;  // warp 12 issues the A/P MMAs, warp 13 the staging loads
constexpr int K1_WU = 6;        // warp 6 issues the W/U MMAs
// staging of one (chunk, head): tiles brought by TMA with 128-byte swizzle, in
// boxes of 128-byte rows (64 bf16 or 32 fp32 channels) of the 64 tokens
constexpr uint32_t S1_STG_K = 0, S1_STG_Q = 16384, S1_STG_V = 32768;  // bf16: 2 boxes of 8 KB
constexpr uint32_t S1_STG_G = 49152;                                  // fp32: 4 boxes of 8 KB
constexpr int LD = 68;                          // fp32 row stride of the 64 x 64 tiles
constexpr uint32_t TILE_BYTES = 64 * LD * 4;    // 17,408
constexpr uint32_t S1_AS = 81920;               // A fp32 [64][LD] (then F^T in its upper blocks)
constexpr uint32_t S1_TS = S1_AS + TILE_BYTES;  // T fp32 [64][LD] (T_RR^T in its upper blocks)
// fp16 K e^g and V, [r][c] 128B-swizzled (MN-major B), side by side: one
// buffer per task parity (the prep of task k + 1 runs while the W/U MMA of
// task k - 1 may still read the other buffer)
constexpr uint32_t S1_KGV1 = 116736;
constexpr uint32_t S1_OPB = 149504;   // tf32 K e^-g: 4 atoms x 64 rows x 128 B
constexpr uint32_t S1_KGV0 = 182272;
constexpr uint32_t S1_TP = 215040;    // fp16 T', K-major SW128 [r][i]
constexpr uint32_t S1_MISC = 223232;
constexpr uint32_t S1_BYTES = S1_MISC + 4096 + 1024;
static_assert(S1_TS + TILE_BYTES <= S1_KGV1 && S1_KGV1 + 32768 <= S1_OPB &&
              S1_OPB + 32768 <= S1_KGV0 && S1_KGV0 + 32768 <= S1_TP && S1_TP + 8192 <= S1_MISC &&
              S1_KGV1 % 1024 == 0 && S1_OPB % 1024 == 0 && S1_KGV0 % 1024 == 0 &&
              S1_TP % 1024 == 0 && S1_BYTES <= 232448, "per-chunk kernel shared-memory layout");
// TMEM: A/P accumulator (64 columns), the tf32 A operand [K e^g ; Q e^g]
// (128 columns, one channel each), W, U~
constexpr int AP_COL = 0, AOP_COL = 128, W_COL = 256, U_COL = 384;
// one N = 256 MMA covers W and U~: their B operands (fp16 K e^g, fp16 V) are
// adjacent 64-column atoms, their accumulators adjacent TMEM columns
static_assert(U_COL == W_COL + 128, "W / U~ accumulators must be adjacent");
constexpr float RANGE_LIMIT = 80.f;                   // e^80 stays inside fp32

struct K1Params {
    CUtensorMap tm_q, tm_k, tm_v, tm_g;   // 3D maps over [T][H][128] (tm_g unused for scalar gates)
    const float *g;                       // scalar gates [T][H] (when scalar_gate)
    const float *beta;
    const int32_t *cu;
    uint8_t *ws;
    int N, H;
    int64_t T;
    int w0, w1;        // chunks [w0, w1) of this launch
    int img0;          // chunk whose operand images sit at the start of the image area
    int scalar_gate;
    int force_timeout;   // fault-injection test build only (see fault_force_timeout)
};

// ---- chain kernel (one 32-column slice per CTA) ------------------------------
constexpr int K2_THREADS = 160;       // warps 0-3: the state, warp 4: MMA and load issue
constexpr int K2_ISSUER = 4;
// K steps of Q^ S issued in round 1 of a chunk; the other five follow P U in
// round 2.  The issuing thread's MMAs run in order, so Q^ S steps queued in
// round 1 delay Kbar^T U, which is on the chain's critical path; behind P U
// they run while the state updates.
constexpr int QS_ROUND1 = 3;
static_assert(QS_ROUND1 >= 1 && QS_ROUND1 <= 8, "P U accumulates onto the round-1 steps of Q^ S");
constexpr uint32_t S2_WQ = 0;          // [W ; Q^] K-major SW128, 2 atoms x 128 rows
constexpr uint32_t S2_KB = 32768;      // Kbar [r][c] SW128 (MN-major A)
constexpr uint32_t S2_PZ = 49152;      // P K-major SW128 (64 rows)
constexpr uint32_t S2_U = 57344;       // U~ slice [64][32] fp16
constexpr uint32_t S2_G = 61440;       // e^gamma_last [128] fp32
constexpr uint32_t S2_STAGE = 62464;   // bytes per stage (multiple of 1024)
constexpr int S2_NSTAGE = 3;           // chunks in flight: loads run two chunks ahead
// S fp16 (K=128 x N=32, MN-major), one buffer per chunk parity: Q^ S steps
// issued after Kbar^T U's commit still read chunk i's S while the state warps
// write chunk i + 1's; the next writer of a buffer (chunk i + 2) waits for
// W S of chunk i + 1, whose commit covers them
constexpr uint32_t S2_SOP = S2_NSTAGE * S2_STAGE;
constexpr uint32_t S2_UOP = S2_SOP + 2 * 8192;            // U fp16, K=64 x N=32, MN-major
constexpr uint32_t S2_MISC = S2_UOP + 4096;
constexpr uint32_t S2_BYTES = S2_MISC + 256 + 1024;
static_assert(S2_PZ + 8192 <= S2_U && S2_U + 4096 <= S2_G && S2_G + 512 <= S2_STAGE &&
              S2_STAGE % 1024 == 0 && S2_PZ % 1024 == 0 && S2_BYTES <= 232448,
              "slice chain shared-memory layout");
constexpr uint32_t S2_TX = 4 * 8192 + 16384 + 8192 + 4096 + 512;   // bytes landing per stage
// TMEM set s (0, 1) at column 128 s: D_W +0 (W S, M = 64), D_O +32 (Q^ S,
// then += P U, M = 64), D_S +64 (Kbar^T U)

struct K2Params {
    const float *S0;
    float *S_T;
    __nv_bfloat16 *o;
    const int32_t *cu;
    uint8_t *ws;
    int N, H;
    int64_t T;
    int w0, w1;        // chunks [w0, w1) of this launch
    int img0;          // chunk whose operand images sit at the start of the image area
    // chunk-affine scan of one sequence (N = 1), see segment_launch_plan
    int nseg;          // 0: off; else the window's chunks in nseg segments
    int seg_len;       // chunks per segment
    int phase;         // 0: segment maps (and segment 0 itself), 1: segments 1..nseg-1
    float *smaps;      // [H][nseg][3][128][128] fp32: M_s, B_s, start state of segment s
    // window plan (many sequences): CTAs take sequences in the plan's order
    // and return at once unless the plan picked their chain form; nullptr:
    // sequence = block index order
    const int32_t *plan;
};

// Roles of a chain CTA in a segment launch.
enum : int { SEG_FULL = 0, SEG_B = 1, SEG_M = 2 };
constexpr int SMAP_M = 0, SMAP_B = 1, SMAP_START = 2;
__host__ __device__ inline float *smap(float *smaps, int nseg, int h, int s, int which) {
    return smaps + ((((size_t)h * nseg + s) * 3 + which) << 14);   // 128 x 128 each
}

// ---- combine step of the chunk-affine scan -----------------------------------
constexpr int COMB_THREADS = 512;
constexpr int SSH_LD = 40;
constexpr uint32_t COMB_BYTES = (128 * 129 + 128 * SSH_LD) * sizeof(float);
// ---- chain kernel, wide form (all 128 columns per CTA) ------------------------
constexpr int K2W_THREADS = 544;       // warps 0-15: the state, warp 16: MMA and load issue
constexpr int K2W_ISSUER = 16;
constexpr uint32_t S2W_WQ = 0;          // [W ; Q^] K-major SW128, 2 atoms x 128 rows
constexpr uint32_t S2W_KB = 32768;      // Kbar [r][c] SW128 (MN-major A)
constexpr uint32_t S2W_PZ = 49152;      // [0 ; P] K-major SW128, 128 rows (rows 0-63 zero)
constexpr uint32_t S2W_U = 65536;       // U~ [4 column blocks][64][32] fp16
constexpr uint32_t S2W_G = 81920;       // e^gamma_last [128] fp32
constexpr uint32_t S2W_STAGE = 82944;   // bytes per stage (multiple of 1024)
constexpr uint32_t S2W_SOP = 2 * S2W_STAGE;   // S fp16, K = 128 x N = 128, MN-major SW128 (2 atoms of 16 KB)
constexpr uint32_t S2W_UOP = S2W_SOP + 32768; // U fp16, K = 64 x N = 128, MN-major SW128 (2 atoms of 8 KB)
constexpr uint32_t S2W_MISC = S2W_UOP + 16384;
constexpr uint32_t S2W_BYTES = S2W_MISC + 256 + 1024;
constexpr uint32_t S2W_TX = 4 * 8192 + 16384 + 8192 + 16384 + 512;   // bytes landing per stage
// TMEM set s (0, 1) at column 256 s: D_A +0 ([W ; Q^] S, then += [0 ; P] U),
// D_S +128 (Kbar^T U)


// ---- kernels -----------------------------------------------------------------
__global__ void __launch_bounds__(1024)
chunk_table_kernel(const int32_t *__restrict__ cu, int N, int64_t T, int cap,
                   int32_t *ws_hdr, int32_t *chunk_base);
__global__ void __launch_bounds__(1024)
window_plan_kernel(const int32_t *__restrict__ chunk_base, int N, int w0, int w1, int H,
                   int slice_cap, int32_t *plan);
__global__ void __launch_bounds__(K1_THREADS, 1) intra_kernel(const __grid_constant__ K1Params p);
__global__ void __launch_bounds__(K2_THREADS, 1) chain_kernel(const K2Params p);
__global__ void __launch_bounds__(K2W_THREADS, 1) chain_wide_kernel(const K2Params p);
__global__ void __launch_bounds__(COMB_THREADS) segment_combine_kernel(float *smaps, int nseg);

}  // namespace tcp
}  // namespace kda
