// kda_prefill_intra.cu -- the per-chunk kernel of the tensor-core prefill
// (layouts and the method overview in kda_prefill_tc.cuh).
#include "kda_prefill_tc.cuh"

namespace kda {
namespace tcp {

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
    // the per-chunk kernel may launch now (it waits for this kernel's
    // completion before reading the table)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// ------------------------------------------------------------------------------
// K1: intra-chunk kernel
// ------------------------------------------------------------------------------
// One CTA per SM walks (chunk, head) tasks, chunk-major, two tasks at a time
// in a software pipeline.  Per task:
//   1. TMA brings k, q, v (bf16) and g (fp32) rows [t0, t0 + 64) of head h
//      into staging, issued as soon as the previous task's prep has consumed
//      the staging tiles.
//   2. Per-channel cumulative log-gate (in place), e^gamma_last, range check.
//   3. Element-wise prep, one token row per thread: tf32 operands
//      [K e^g ; Q e^g] (into TMEM) and K e^-g for A / P, fp16 K e^g and V for
//      W / U~ (one buffer per task parity), the Q^ and Kbar workspace images.
//   4. One M = 128 tf32 MMA group (16 K steps): rows 0-63 give A / beta,
//      rows 64-127 give P.  A chunk whose decay exceeds e^80 on some channel
//      would overflow those factors, so it takes an exact pairwise CUDA-core
//      path instead.
//   5. A / P leave TMEM (A to shared memory, P to the workspace image), then
//      T = (I + A)^-1 on CUDA cores by warps 0-5 (fp32, 16 x 16 blocks,
//      register-tiled block forward substitution), written as the fp16 image
//      of T' = T Diag(beta).
//   6. W = T' (K e^g), U~ = T' V on tcgen05 (fp16), moved from TMEM to the
//      workspace before the next task's inverse.
// Steps 2-4 of task k + 1 run on warps 8-15 while warps 0-7 first move task
// k - 1's W and U~ out and warps 0-5 then run the inverse of task k.  Warp
// 12 issues the A/P MMAs, warp 13 the staging loads and warp 6 the W/U MMAs,
// each from one elected lane.  The inverse then hides the prep's latency
// instead of adding to it.
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
// Scratch: two 64 x LD fp32 tiles.  A (lower blocks) and T (diagonal and
// lower blocks) keep their strictly upper blocks free, so F_RI^T goes to A's
// upper block (I, R) and T_RR^T to one upper block of T (tt_block).
constexpr int INV_THREADS = 192;
__device__ __forceinline__ float *tt_block(float *Ts, int R) {
    // R = 0..3 -> blocks (0, 2), (0, 1), (1, 2), (2, 3) of T
    return Ts + (16 * (R == 0 ? 0 : R - 1)) * LD + 16 * (R == 0 ? 2 : R);
}
__device__ __forceinline__ void invert_unit_lower(float *As, float *Ts, const float *sB,
                                                  uint8_t *tp_img, int tid) {
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
        float4 *trow = reinterpret_cast<float4 *>(tt_block(Ts, R) + j * LD);
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
        mm16_2x4(f, tt_block(Ts, R) + m0, As + (16 * R) * LD + 16 * I + n0);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            *reinterpret_cast<float2 *>(As + (16 * I + n0 + e) * LD + 16 * R + m0) =
                make_float2(f[0][e], f[1][e]);
    }
    bar_sync(1, INV_THREADS);
    float acc[2][4] = {};
#pragma unroll
    for (int pass = 0; pass < 3; ++pass) {
        const int J = I + pass;
        if (J < R) {
            mm16_2x4(acc, As + (16 * J) * LD + 16 * R + m0, Ts + (16 * J) * LD + 16 * I + n0);
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
    float *sB2 = eL + 128;                                 // [2][64] beta, by task parity
    float *tot = sB2 + 128;                                // [2][128] scan segment totals
    float *sGs = tot + 256;                                // [64] scalar gates (scalar_gate)
    int32_t *sflag = reinterpret_cast<int32_t *>(sGs + 64);   // [2] out-of-range chunk, by parity
    // [0] TMA, [1] A/P, [2] W/U, [3] [4] drains of the two MMA issuers
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sflag + 2);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mbar + 5);
    float *As = reinterpret_cast<float *>(sm + S1_AS);
    float *Ts = reinterpret_cast<float *>(sm + S1_TS);

    const int tid = threadIdx.x, lane = tid & 31;
    // warp index the compiler knows to be warp-uniform, so that an issuing
    // warp's branch keeps the MMA operands in uniform registers
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
    const int lt = tid - 256;            // index within warps 8-15 (the prep group)
    int32_t *ws_hdr = reinterpret_cast<int32_t *>(p.ws);
    const int32_t *chunk_base = reinterpret_cast<const int32_t *>(p.ws + WS_HEADER);
    uint8_t *img_base = p.ws + ws_images_offset(p.N);
    const int H = p.H;

    if (tid == 0) {
        mbar_init(&mbar[0], 1);
        mbar_init(&mbar[1], 1);   // A/P MMAs
        mbar_init(&mbar[2], 1);   // W and U~ MMAs
        mbar_init(&mbar[3], 1);   // drains after a failed wait
        mbar_init(&mbar[4], 1);
        mbar_fence_init();
    }
#ifdef KDA_FAULT_INJECTION
    // Fault-injection test build: wait on the load barrier before any load has
    // been issued (nothing will arrive), before TMEM is allocated and before
    // any MMA, so the bounded wait gives up with nothing in flight; the CTA
    // records the timeout and returns.
    if (p.force_timeout) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        __syncthreads();
        if (!__syncthreads_and(mbar_wait(&mbar[0], 0, 64))) {
            if (tid == 0) ws_fail(ws_hdr, 1);
            return;
        }
    }
#endif
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
    // This kernel may run as the chunk table's programmatic dependent: the
    // setup above overlaps it, and its results (the chunk offsets, the status
    // word it clears) are read after its completion.  The chain kernel that
    // follows may then launch: its CTAs take SMs as this kernel's CTAs
    // finish, and wait for this kernel's completion before reading its
    // results.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int total = chunk_base[p.N];
    const int c_end = min(p.w1, total);
    const int ntask = (c_end > p.w0 ? c_end - p.w0 : 0) * H;
    const int stride = gridDim.x;
    // this CTA's tasks: k = 0 .. n - 1 is task blockIdx.x + k * stride
    const int n = (int)blockIdx.x < ntask ? (ntask - (int)blockIdx.x + stride - 1) / stride : 0;
    auto task_of = [&](int k) { return (int)blockIdx.x + k * stride; };
    auto img_of = [&](int k) {
        return img_base + ((uint64_t)(p.w0 - p.img0) * H + (uint64_t)task_of(k)) * CH_STRIDE;
    };

    struct Pos { int h, L; int64_t t0; };
    // A task's position in two steps: fetch issues the offset-table loads,
    // finish is their first use (placed an iteration later, so that the loads'
    // latency is hidden).  Together they give the sequence bounds clamped into
    // [0, T] (as seq_bounds does) and the chunk's first token and length.
    struct PosRaw { int ch, h; int32_t c0, c1, cb; };
    auto pos_fetch = [&](int k) {
        PosRaw r{-1, 0, 0, 0, 0};
        if (k >= n) return r;
        const int task = task_of(k);
        r.ch = p.w0 + task / H;
        r.h = task % H;
        const int sq = find_seq(chunk_base, p.N, r.ch);
        r.c0 = p.cu[sq];
        r.c1 = p.cu[sq + 1];
        r.cb = chunk_base[sq];
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
    // beta (and the scalar gate) of row lt of task k, read ahead into registers
    auto row_params = [&](const Pos &q, int k, float &b, float &gs) {
        b = 0.f; gs = 0.f;
        if (lt >= 0 && lt < C && k < n && lt < q.L) {
            b = p.beta[(q.t0 + lt) * H + q.h];
            if (p.scalar_gate) gs = p.g[(q.t0 + lt) * H + q.h];
        }
    };
    constexpr uint32_t TILE_BF16 = 16384, TILE_G = 32768;
    // the staging loads of one task (one thread)
    auto issue_tma = [&](const Pos &q) {
        mbar_arrive_expect_tx(&mbar[0], 3 * TILE_BF16 + (p.scalar_gate ? 0 : TILE_G));
        // boxes of 128 bytes of channels: two per bf16 tile, four per fp32 tile
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            tma_load_3d(sm + S1_STG_K + 8192 * b, &p.tm_k, 64 * b, q.h, (int)q.t0, &mbar[0]);
            tma_load_3d(sm + S1_STG_Q + 8192 * b, &p.tm_q, 64 * b, q.h, (int)q.t0, &mbar[0]);
            tma_load_3d(sm + S1_STG_V + 8192 * b, &p.tm_v, 64 * b, q.h, (int)q.t0, &mbar[0]);
        }
        if (!p.scalar_gate) {
#pragma unroll
            for (int b = 0; b < 4; ++b)
                tma_load_3d(sm + S1_STG_G + 8192 * b, &p.tm_g, 32 * b, q.h, (int)q.t0, &mbar[0]);
        }
    };
    // W (or U~) of a finished task: the 16 rows of this warp's lane quadrant
    // (row r of the M = 64 accumulators sits in lane r % 16 of quadrant r / 16)
    auto drain_half = [&](uint8_t *dst, bool is_u) {
        const int r = 16 * (warp & 3) + lane;
        const uint32_t col0 = is_u ? U_COL : W_COL;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
            float x[2][16];
            tmem_ld16(tmem_at(tmem, warp, col0 + c), x[0]);
            tmem_ld16(tmem_at(tmem, warp, col0 + c + 16), x[1]);
            tmem_wait_ld();
            if (lane < 16) {
#pragma unroll
                for (int hc = 0; hc < 4; ++hc) {
                    const int c0 = c + 8 * hc;
                    const uint4 v = pack8_h(x[hc >> 1] + 8 * (hc & 1));
                    if (is_u)
                        *reinterpret_cast<uint4 *>(dst + IMG_U + (c0 >> 5) * 4096 +
                                                   u_img_off(r, (c0 & 31) >> 3)) = v;
                    else
                        *reinterpret_cast<uint4 *>(dst + IMG_W + rc_img_off(r, c0)) = v;
                }
            }
        }
    };

    // Task k passes through: stage P (iteration k - 1: gate scan and prep by
    // warps 8-15, then the A/P MMA), stage I (iteration k: A/P readout by all
    // warps, then task k - 1's W/U drain and the inverse by warps 0-7 / 0-5
    // while warps 8-15 run stage P of task k + 1; then the W/U MMA), and its
    // W and U~ leave TMEM at the start of iteration k + 1's stage I part 2.  Positions: p0 = task i, pA = i + 1, pB = i + 2, rC = i + 3.
    Pos p0{0, 0, 0}, pA = pos_finish(pos_fetch(0)), pB = pos_finish(pos_fetch(1));
    PosRaw rC = pos_fetch(2);
    float b_reg, gs_reg;
    row_params(pA, 0, b_reg, gs_reg);
    int last_tma = -1;      // the last task whose staging loads were issued (uniform)
    if (n > 0) {
        if (tid == 0) issue_tma(pA);
        last_tma = 0;
    }
    bool ok = true, bad = false;
    uint32_t ap_it = 0;     // A/P MMAs waited for (uniform)
    int i = -1;
    for (; i < n; ++i) {
        // ---- stage I, part 1: A and P of task i ------------------------------
        if (i >= 0) {
            const bool slow_i = __shfl_sync(0xffffffffu, sflag[i & 1], 0) != 0;
            uint8_t *out_i = img_of(i);
            const float *sBi = sB2 + 64 * (i & 1);
            if (!slow_i) {
                fence_before_sync();
                ok = __syncthreads_and(!bad && mbar_wait(&mbar[1], ap_it & 1));
                ++ap_it;
                fence_after_sync();
                if (!ok) break;
                // warp = (lane quadrant q, 16-column block cb); lane = row
                const int q = warp & 3, cb = warp >> 2;
                const int row = 32 * q + lane;
                float d[16];
                tmem_ld16(tmem_at(tmem, q, AP_COL + 16 * cb), d);
                tmem_wait_ld();
                if (row < 64) {
                    const float b = sBi[row];
                    float4 *arow = reinterpret_cast<float4 *>(As + row * LD + 16 * cb);
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                        float a4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = 16 * cb + 4 * e4 + e;
                            a4[e] = row > c ? b * d[4 * e4 + e] : 0.f;
                        }
                        arow[e4] = make_float4(a4[0], a4[1], a4[2], a4[3]);
                    }
                } else {
                    const int r = row - 64;
                    float pv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) pv[e] = (16 * cb + e) <= r ? d[e] : 0.f;
                    *reinterpret_cast<uint4 *>(out_i + IMG_P + sw128_off(r, 2 * cb)) = pack8_h(pv);
                    *reinterpret_cast<uint4 *>(out_i + IMG_P + sw128_off(r, 2 * cb + 1)) = pack8_h(pv + 8);
                }
            } else {
                // ---- exact pairwise path for chunks whose decay leaves fp32
                // range (their staging is still in place: the next task's
                // loads wait for this)
                const int L = p0.L;
                auto kq = [&](uint32_t tile, int t, int c) {
                    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                        sm + tile + stg16_off(t, c)));
                };
                auto gm = [&](int t, int c) {
                    return *reinterpret_cast<const float *>(sm + S1_STG_G + stg32_off(t, c));
                };
                for (int e = tid; e < C * C; e += K1_THREADS) {
                    const int r = e >> 6, c2 = e & 63;
                    float a = 0.f, pp = 0.f;
                    if (c2 <= r && r < L) {
                        for (int c = 0; c < D; ++c) {
                            const float ki = kq(S1_STG_K, c2, c) * __expf(gm(r, c) - gm(c2, c));
                            a += kq(S1_STG_K, r, c) * ki;
                            pp += kq(S1_STG_Q, r, c) * ki;
                        }
                    }
                    As[r * LD + c2] = c2 < r ? sBi[r] * a : 0.f;
                    *reinterpret_cast<__half *>(out_i + IMG_P + sw128_off(r, c2 >> 3) + (c2 & 7) * 2) =
                        __float2half_rn(pp);
                }
                fence_before_sync();
                __syncthreads();
                if (i + 1 < n) {      // staging is consumed
                    if (tid == 0) issue_tma(pA);
                    last_tma = i + 1;
                }
            }
        }
        __syncthreads();

        // ---- stage I, part 2 (task i) beside stage P (task i + 1) ------------
        if (warp < 8) {
            if (i >= 0) {
                // task i - 1's W and U~ leave TMEM first (W by warps 0-3, U~ by
                // warps 4-7, one lane quadrant each), once its W/U MMA has
                // completed: their stores then run beside the gate scan, the
                // inverse beside the prep
                if (i >= 1) {
                    if (!mbar_wait(&mbar[2], (uint32_t)((i - 1) & 1))) bad = true;
                    fence_after_sync();
                    drain_half(img_of(i - 1), warp >= 4);
                }
                // T = (I + A)^-1 of task i; its fp16 T' replaces task i - 1's
                // in the W/U A operand, which that MMA no longer reads
                if (warp < 6) {
                    invert_unit_lower(As, Ts, sB2 + 64 * (i & 1), sm + S1_TP, tid);
                    fence_async_smem();
                }
            }
        } else if (i + 1 < n) {
            const int k = i + 1;
            uint8_t *out = img_of(k);
            const int L = pA.L;
            const bool need_wu = k >= 2;   // W/U MMA of task k - 2 reads this B buffer
            const uint32_t kgv = (k & 1) ? S1_KGV1 : S1_KGV0;
            if (lt < C) {
                sB2[64 * (k & 1) + lt] = b_reg;
                sGs[lt] = gs_reg;
            }
            if (lt == 0) sflag[k & 1] = 0;
            row_params(pB, k + 1, b_reg, gs_reg);   // consumed next iteration
            if (!mbar_wait(&mbar[0], (uint32_t)(k & 1))) bad = true;
            if (need_wu && !mbar_wait(&mbar[2], (uint32_t)((k - 2) & 1))) bad = true;
            if (L < C) {
                // the chunk ends inside the tile: rows L..63 become no-op tokens
                // (k = q = v = 0, g = 0; beta is already 0 there), so that the
                // scan and the prep need no per-row test
                // (a token row is one 128-byte line in each of the ten boxes)
                const int nrow = C - L;
                for (int e = lt; e < nrow * 80; e += 256) {
                    const int r = L + e / 80, bx = (e % 80) >> 3, x = e & 7;
                    const uint32_t box = bx < 2 ? S1_STG_K + 8192 * bx
                                       : bx < 4 ? S1_STG_Q + 8192 * (bx - 2)
                                       : bx < 6 ? S1_STG_V + 8192 * (bx - 4)
                                                : S1_STG_G + 8192 * (bx - 6);
                    *reinterpret_cast<uint4 *>(sm + box + (r >> 3) * 1024 + (r & 7) * 128 + x * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            bar_sync(2, 256);

            // cumulative log-gate, in place (rows past the sequence: g = 0);
            // thread = (channel c, 32-row segment sg)
            {
                const int c = lt & 127, sg = lt >> 7;
                auto G = [&](int r) -> float & {
                    return *reinterpret_cast<float *>(sm + S1_STG_G + stg32_off(r, c));
                };
                float v[32];
                if (p.scalar_gate) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = sGs[32 * sg + j];
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = G(32 * sg + j);
                }
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    acc += v[j];
                    v[j] = acc;
                }
                tot[sg * 128 + c] = acc;
                bar_sync(2, 256);
                const float off = sg ? tot[c] : 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) G(32 * sg + j) = v[j] + off;
                if (sg == 1) {
                    gL[c] = acc + off;
                    eL[c] = __expf(acc + off);
                    if (-(acc + off) > RANGE_LIMIT) sflag[k & 1] = 1;
                }
            }
            bar_sync(2, 256);
            const bool slow = __shfl_sync(0xffffffffu, sflag[k & 1], 0) != 0;

            // element-wise prep, one token row per thread: warp w owns TMEM
            // lane quadrant w % 4 -- rows 32 (w % 4) .. + 31 of the M = 128 A
            // operand [K e^g ; Q e^g] -- and channels 64 ((w - 8) / 4) .. + 63,
            // in four passes of 16.  K rows (lanes 0-63, token t = lane):
            // K e^g into the TMEM operand and the fp16 W operand, V into the
            // fp16 U~ operand.  Q rows (lanes 64-127, token t = lane - 64):
            // Q e^g into the TMEM operand and the Q^ image, and for the same
            // token K e^-g (the tf32 B operand of A / P, not on the slow path)
            // and the Kbar image.  A warp's 32 lanes read and write 32
            // consecutive token rows at one 16-byte chunk position, which the
            // 128-byte swizzle spreads over all banks.
            const int quad = warp & 3;
            const int rr = 32 * quad + lane;
            const bool krow = rr < 64;
            const int t = krow ? rr : rr - 64;
#pragma unroll 1
            for (int cqi = 0; cqi < 2; ++cqi) {
                const int cq = 2 * ((warp - 8) >> 2) + cqi;
                float aop[32];
#pragma unroll
                for (int hp = 0; hp < 2; ++hp) {
                    const int c0 = 32 * cq + 16 * hp;        // first channel of this pass
                    float gm[16], x[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 g4 = *reinterpret_cast<const float4 *>(
                            sm + S1_STG_G + stg32_off(t, c0 + 4 * j));
                        gm[4 * j] = g4.x; gm[4 * j + 1] = g4.y; gm[4 * j + 2] = g4.z; gm[4 * j + 3] = g4.w;
                    }
                    auto load16 = [&](uint32_t tile, float (&dst)[16]) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const uint4 raw = *reinterpret_cast<const uint4 *>(
                                sm + tile + stg16_off(t, c0 + 8 * j));
                            const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = __bfloat1622float2(b2[e]);
                                dst[8 * j + 2 * e] = f.x;
                                dst[8 * j + 2 * e + 1] = f.y;
                            }
                        }
                    };
                    load16(krow ? S1_STG_K : S1_STG_Q, x);
#pragma unroll
                    for (int e = 0; e < 16; ++e) aop[16 * hp + e] = x[e] * __expf(gm[e]);
                    if (krow) {
                        // fp16 K e^g: B operand of W = T' (K e^g)
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            *reinterpret_cast<uint4 *>(sm + kgv + rc_img_off(t, c0 + 8 * j)) =
                                pack8_h(aop + 16 * hp + 8 * j);
                        // fp16 V: B operand of U~ = T' V
                        load16(S1_STG_V, x);
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            *reinterpret_cast<uint4 *>(sm + kgv + 16384 + rc_img_off(t, c0 + 8 * j)) =
                                pack8_h(x + 8 * j);
                    } else {
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            *reinterpret_cast<uint4 *>(out + IMG_Q + rc_img_off(t, c0 + 8 * j)) =
                                pack8_h(aop + 16 * hp + 8 * j);
                        // K e^-g and Kbar = K e^(gamma_last - gamma) of token t
                        load16(S1_STG_K, x);
                        float kb[16];
                        if (!slow) {   // e^-gamma <= e^80 here: Kbar = (K e^-g) e^gamma_last
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                x[e] *= __expf(-gm[e]);
                                kb[e] = x[e] * eL[c0 + e];
                            }
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                *reinterpret_cast<float4 *>(sm + S1_OPB + cq * 8192 +
                                                            sw128_off(t, 4 * hp + j)) =
                                    make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) kb[e] = x[e] * __expf(gL[c0 + e] - gm[e]);
                        }
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            *reinterpret_cast<uint4 *>(out + IMG_KT + rc_img_off(t, c0 + 8 * j)) =
                                pack8_h(kb + 8 * j);
                    }
                }
                tmem_st32(tmem_at(tmem, quad, AOP_COL + 32 * cq), aop);
            }
            if (lt < 128) reinterpret_cast<float *>(out + IMG_G)[lt] = eL[lt];
            tmem_wait_st();
            fence_async_smem();
            // the prep group is done with the staging and the A / P operands:
            // warp 12 starts task k's A/P MMA and, beside it, warp 13 task
            // k + 1's staging loads (a chunk out of range keeps its staging
            // for the pairwise path, which issues the loads itself)
            fence_before_sync();
            bar_sync(2, 256);
            if (warp == K1_ISSUER0) {
                fence_after_sync();
                const uint32_t ap_acc = warp_uniform(tmem + AP_COL);
                const uint32_t ap_aop = warp_uniform(tmem + AOP_COL);
                const uint64_t ap_db = sdesc_k_sw128(warp_uniform(smem_addr(sm)) + S1_OPB);
                if (elect_one() && !slow) {
                    constexpr uint32_t id = idesc(128, 64, FMT_TF32, FMT_TF32, 0, 0);
#pragma unroll
                    for (int s2 = 0; s2 < 16; ++s2)   // channel atom s2 / 4 of the B operand
                        mma_tf32_tmem_a(ap_acc, ap_aop + 8 * s2,
                                        sdesc_add(ap_db, (s2 >> 2) * 8192 + (s2 & 3) * 32), id, s2 > 0);
                    mma_commit(&mbar[1]);
                }
                __syncwarp();
            } else if (warp == K1_ISSUER0 + 1) {
                if (elect_one() && !slow && k + 1 < n) issue_tma(pB);
                __syncwarp();
            }
        }
        fence_before_sync();
        ok = __syncthreads_and(!bad);
        fence_after_sync();
        // task i + 2's staging loads left with the A/P MMA unless task i + 1 is
        // out of range: counted before a possible exit, which waits for them
        const bool slow_n = i + 1 < n && __shfl_sync(0xffffffffu, sflag[(i + 1) & 1], 0) != 0;
        if (i + 2 < n && !slow_n) last_tma = i + 2;
        if (!ok) break;

        // ---- W/U MMA of task i (warp 6's elected lane; warp 12 meanwhile
        // joins the A/P wait)
        if (warp == K1_WU && i >= 0) {
            const uint32_t smb = warp_uniform(smem_addr(sm));
            const uint32_t wu_acc = warp_uniform(tmem + W_COL);
            const uint64_t wu_dt = sdesc_k_sw128(smb + S1_TP);
            if (elect_one()) {
                // [W | U~] = T' [K e^g | V] (fp16, M = 64, N = 256: the two B
                // operands sit side by side as four 64-column MN-major atoms,
                // and the accumulators side by side in TMEM)
                const uint64_t wu_db = sdesc(smb + ((i & 1) ? S1_KGV1 : S1_KGV0), 8192, 1024,
                                             LAYOUT_SW128);
                constexpr uint32_t id = idesc(64, 256, FMT_F16, FMT_F16, 0, 1);
#pragma unroll
                for (int s2 = 0; s2 < 4; ++s2)
                    mma_f16(wu_acc, sdesc_add(wu_dt, 32 * s2), sdesc_add(wu_db, 2048 * s2), id, s2 > 0);
                mma_commit(&mbar[2]);
            }
            __syncwarp();
        }
        p0 = pA;
        pA = pB;
        pB = pos_finish(rC);
        rC = pos_fetch(i + 4);
    }
    // the last W/U MMA, then its results
    if (ok && n > 0) {
        if (warp < 8) {
            if (!mbar_wait(&mbar[2], (uint32_t)((n - 1) & 1))) bad = true;
            fence_after_sync();
            drain_half(img_of(n - 1), warp >= 4);
        }
        ok = __syncthreads_and(!bad);
    }
    if (!ok) {
        if (tid == 0) {
            ws_fail(ws_hdr, 1);
            // let copies still in flight finish before the CTA's shared memory
            // is released (at most one set of staging loads is in flight)
            if (last_tma >= 0) mbar_wait(&mbar[0], (uint32_t)(last_tma & 1), 1u << 20);
        }
        if (warp == K1_ISSUER0 || warp == K1_WU) {   // and the MMAs, before TMEM is released
            uint64_t *mb = &mbar[warp == K1_WU ? 4 : 3];
            if (elect_one()) {
                mma_commit(mb);
                mbar_wait(mb, 0, 1u << 20);
            }
            __syncwarp();
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc<512>(tmem);
}

}  // namespace tcp
}  // namespace kda
