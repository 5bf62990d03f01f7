// kda_prefill_chain.cu -- the state chain of the tensor-core prefill: the
// slice form, the combine step of the chunk-affine scan and the wide form
// (layouts and the method overview in kda_prefill_tc.cuh).
#include "kda_prefill_tc.cuh"

namespace kda {
namespace tcp {

// ------------------------------------------------------------------------------
// K2: chain kernel
// ------------------------------------------------------------------------------
// One CTA of 160 threads per (sequence, head, block of 32 state columns):
// warps 0-3 hold the fp32 state (thread t = row t, a dk channel), warp 4
// issues the MMAs and the operand loads.  Per chunk:
//   round 1: D_W = W S (M = 64), then part of D_O = Q^ S (M = 64)
//   U = U~ - W S (fp16);
//   round 2: D_S = Kbar^T U, then D_O += P U and the rest of Q^ S (D_O then
//   holds O)
//   S = Diag(e^gamma_last) S + D_S.
// (The wide form below, one CTA per (sequence, head), keeps one M = 128
// [W ; Q^] S and [0 ; P] U.)
// TMEM accumulators alternate between two sets so that the outputs of chunk
// i are read while the MMAs of chunk i + 1 run; operand images arrive with
// bulk async copies two chunks ahead (three stages).
// ------------------------------------------------------------------------------
// window plan (batches of many sequences): the sequences with chunks in the
// window [w0, w1) -- and, in the first window, the empty ones, whose initial
// state passes through -- ordered by their chain length in the window, longest
// first (a counting sort over the length, at most WINDOW_CHUNKS).  A chain
// CTA runs for a time proportional to its length, so starting the longest
// first shortens the tail of the launch (longest-processing-time-first list
// scheduling); the chain form follows from the number of chain slices listed.
// ------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
window_plan_kernel(const int32_t *__restrict__ chunk_base, int N, int w0, int w1, int H,
                   int slice_cap, int32_t *plan) {
    constexpr int NB = WINDOW_CHUNKS + 1;   // bin WINDOW_CHUNKS - length, length 0 .. WINDOW_CHUNKS
    __shared__ int32_t start[NB];
    __shared__ int32_t warp_tot[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < NB; i += 1024) start[i] = 0;
    __syncthreads();
    for (int n = tid; n < N; n += 1024) {
        const int cb = chunk_base[n], ce = chunk_base[n + 1];
        const int len = min(max(0, min(ce, w1) - max(cb, w0)), WINDOW_CHUNKS);
        if (len > 0 || (w0 == 0 && cb == ce)) atomicAdd(&start[WINDOW_CHUNKS - len], 1);
    }
    __syncthreads();
    // exclusive scan of the bins: thread t owns bins 2t and 2t + 1, thread 1023
    // also the last bin
    const int b0 = 2 * tid;
    const int c0 = start[b0], c1 = start[b0 + 1], c2 = tid == 1023 ? start[NB - 1] : 0;
    int x = c0 + c1 + c2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    const int excl = x - (c0 + c1 + c2) + (warp > 0 ? warp_tot[warp - 1] : 0);
    start[b0] = excl;
    start[b0 + 1] = excl + c0;
    if (tid == 1023) {
        start[NB - 1] = excl + c0 + c1;
        const int total = excl + c0 + c1 + c2;
        plan[1] = total;
        plan[0] = (int64_t)total * H * NSLICE > slice_cap ? PLAN_WIDE : PLAN_SLICE;
    }
    __syncthreads();
    for (int n = tid; n < N; n += 1024) {
        const int cb = chunk_base[n], ce = chunk_base[n + 1];
        const int len = min(max(0, min(ce, w1) - max(cb, w0)), WINDOW_CHUNKS);
        if (len > 0 || (w0 == 0 && cb == ce)) plan[2 + atomicAdd(&start[WINDOW_CHUNKS - len], 1)] = n;
    }
}

__global__ void __launch_bounds__(K2_THREADS, 1) chain_kernel(const K2Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    // [0..2] loads of the three stages, [3] W S, [4] Kbar^T U, [5..6] the
    // outputs of TMEM set 0 / 1 (their P U), [7] drain
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + S2_MISC);
    constexpr int MB_R1 = S2_NSTAGE, MB_R2S = MB_R1 + 1, MB_R2O = MB_R1 + 2, MB_DRAIN = MB_R1 + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mbar + MB_DRAIN + 1);
    int32_t *iss = reinterpret_cast<int32_t *>(tmem_slot + 1);   // [3] last chunk loaded per stage

    const int tid = threadIdx.x, lane = tid & 31;
    // warp index the compiler knows to be warp-uniform (so that the issuer
    // warp's branch keeps the MMA operands in uniform registers)
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
    const bool issuer = warp == K2_ISSUER;   // MMAs and operand loads; holds no state
    const int row = tid;                     // warps 0-3: state row (dk channel) = TMEM lane
    const int H = p.H;
    const int unit = blockIdx.x;
    int slice = unit % NSLICE;
    int h = (unit / NSLICE) % H;
    int n = unit / (NSLICE * H);
    // This kernel may run as the per-chunk kernel's programmatic dependent:
    // its CTAs then start while that kernel's last CTAs still run.  They wait
    // for its completion here, before the first global read of anything this
    // call wrote (the chunk table, a previous window's final states, the
    // images, the status word): the wait orders the writes of the kernels
    // before it for this grid, and nothing else does.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (p.plan) {   // many sequences: the window plan's order, if it picked this form
        if (p.plan[0] != PLAN_SLICE || unit >= p.plan[1] * H * NSLICE) return;
        n = p.plan[2 + unit / (NSLICE * H)];
    }
    int32_t *ws_hdr = reinterpret_cast<int32_t *>(p.ws);
    const int32_t *chunk_base = reinterpret_cast<const int32_t *>(p.ws + WS_HEADER);
    const uint8_t *img_base = p.ws + ws_images_offset(p.N);
    // A per-chunk kernel of this call that gave up on a wait left its images
    // incomplete: o and S_T stay untouched (the status reports it).
    auto upstream_failed = [&]() { return *reinterpret_cast<volatile int32_t *>(ws_hdr) != 0; };

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
    const int64_t sbase_g = ((int64_t)n * H + h) * D * D + (int64_t)row * D + slice * DVS;
    if (cb == ce && !p.nseg) {            // empty sequence: pass the state through
        if (upstream_failed()) return;
        if (p.w0 == 0 && !issuer) {
            for (int j = 0; j < DVS; j += 4) {
                float4 x = p.S0 ? *reinterpret_cast<const float4 *>(p.S0 + sbase_g + j)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4 *>(p.S_T + sbase_g + j) = x;
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
        for (int j = 0; j < DVS; ++j) S[j] = (row == slice * DVS + j) ? 1.f : 0.f;
    } else if (role == SEG_B || issuer) {
#pragma unroll
        for (int j = 0; j < DVS; ++j) S[j] = 0.f;
    } else {
        const float *src = (a == cb) ? p.S0 : p.S_T;
        int64_t off = sbase_g;
        if (p.nseg && seg > 0) {  // the start state the combine step produced
            src = smap(p.smaps, p.nseg, h, seg, SMAP_START);
            off = (int64_t)row * D + slice * DVS;
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
    if (tid == 0) {
        for (int j = 0; j <= MB_DRAIN; ++j) mbar_init(&mbar[j], 1);
        mbar_fence_init();
        for (int j = 0; j < S2_NSTAGE; ++j) iss[j] = -1;
    }
    if (warp == 0) tmem_alloc<256>(tmem_slot);
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = warp_uniform(*tmem_slot);
    const uint32_t smb = warp_uniform(smem_addr(sm));
    if (upstream_failed()) {
        fence_before_sync();
        __syncthreads();
        if (warp == 0) tmem_dealloc<256>(tmem);
        return;
    }

    auto issue_loads = [&](int ch, int stage) {
        const uint8_t *src = img_base + ((uint64_t)(ch - p.img0) * H + h) * CH_STRIDE;
        uint8_t *dst = sm + stage * S2_STAGE;
        uint64_t *mb = &mbar[stage];
        iss[stage] = ch - a;
        mbar_arrive_expect_tx(mb, S2_TX);
        bulk_g2s(dst + S2_WQ, src + IMG_W, 8192, mb);              // W, k 0-63
        bulk_g2s(dst + S2_WQ + 8192, src + IMG_Q, 8192, mb);       // Q^, k 0-63
        bulk_g2s(dst + S2_WQ + 16384, src + IMG_W + 8192, 8192, mb);
        bulk_g2s(dst + S2_WQ + 24576, src + IMG_Q + 8192, 8192, mb);
        bulk_g2s(dst + S2_KB, src + IMG_KT, 16384, mb);
        bulk_g2s(dst + S2_PZ, src + IMG_P, 8192, mb);
        bulk_g2s(dst + S2_U, src + IMG_U + slice * 4096, 4096, mb);
        bulk_g2s(dst + S2_G, src + IMG_G, 512, mb);
    };
    if (issuer) {                 // chunks a and a + 1 up front
        if (elect_one()) {
            if (a < b) issue_loads(a, 0);
            if (a + 1 < b) issue_loads(a + 1, 1);
        }
        __syncwarp();
    }

    const uint32_t id_m64 = idesc(64, DVS, FMT_F16, FMT_F16, 0, 1);   // W S, Q^ S, P U
    const uint32_t id_kb = idesc(128, DVS, FMT_F16, FMT_F16, 1, 1);

    // Half (16 columns) of the O rows of a finished chunk, once its P U MMA
    // (the last to accumulate into them) has completed: row r = 16 warp + lane
    // of the M = 64 accumulator sits in lane r % 16 of quadrant r / 16 (lanes
    // 0-15 store).
    auto store_o = [&](int set, int64_t t0, int L, uint32_t pu_parity, int half) -> bool {
        if (!mbar_wait(&mbar[MB_R2O + set], pu_parity)) return false;
        fence_after_sync();
        float oa[16];
        tmem_ld16(tmem_at(tmem, warp, 128 * set + 32 + 16 * half), oa);
        tmem_wait_ld();
        const int r = 16 * warp + lane;
        if (lane < 16 && r < L) {
            __nv_bfloat16 *dst = p.o + ((t0 + r) * H + h) * D + slice * DVS + 16 * half;
#pragma unroll
            for (int gq = 0; gq < 2; ++gq) {
                const float *src = oa + 8 * gq;
                __nv_bfloat162 b0 = __floats2bfloat162_rn(src[0], src[1]);
                __nv_bfloat162 b1 = __floats2bfloat162_rn(src[2], src[3]);
                __nv_bfloat162 b2 = __floats2bfloat162_rn(src[4], src[5]);
                __nv_bfloat162 b3 = __floats2bfloat162_rn(src[6], src[7]);
                *reinterpret_cast<uint4 *>(dst + 8 * gq) = make_uint4(
                    *reinterpret_cast<uint32_t *>(&b0), *reinterpret_cast<uint32_t *>(&b1),
                    *reinterpret_cast<uint32_t *>(&b2), *reinterpret_cast<uint32_t *>(&b3));
            }
        }
        return true;
    };

    // Per chunk i (stage i % 3, TMEM set i % 2: D_W = set columns 0-31 (W S,
    // M = 64), D_O = columns 32-63 (Q^ S + P U, M = 64), D_S = columns 64-95
    // (Kbar^T U, M = 128)).  Warps 0-3 hold the fp32 state (thread = row);
    // warp 4 issues every MMA and load from its elected lane, so no
    // state-holding warp ever blocks on an issue:
    //   B1 (all):       S (fp16 operand) written, chunk i's operands landed
    //   warp 4:         D_W = W S (8 K steps, M = 64: half the operand reads
    //                   of the M = 128 [W ; Q^] S, and on the critical path)
    //                   -> MB_R1, then the first QS_ROUND1 K steps of
    //                   D_O = Q^ S, then the operands of chunk i + 2 into the
    //                   stage of chunk i - 1 (once chunk i - 1's P U is done)
    //   warps 0-3:      half the O rows of chunk i - 1 (while W S runs), then
    //                   U = U~ - W S (token rows 16 warp + lane, lanes 0-15)
    //   B2 (all):       U written
    //   warp 4:         D_S = Kbar^T U (4 K steps) -> MB_R2S, then
    //                   D_O += P U (4 K steps, M = 64) and the rest of Q^ S
    //                   -> MB_R2O of the set
    //   warps 0-3:      the other half (while Kbar^T U runs), then
    //                   S = Diag(e^gamma_last) S + D_S   (after MB_R2S)
    // W S of chunk i completes after every MMA of chunk i - 1 (one issuing
    // thread, whose commits track all its earlier MMAs), so when B2 passes,
    // the U operand's previous contents are free.  The output barrier of a
    // set completes once every two chunks, and its waiters (the issuer before
    // the loads, warps 0-3 before the O rows) wait for it before B2 of the
    // next chunk, whose P U completes its next phase.  Loads run two chunks
    // ahead.
    bool ok = true, bad = false;
    int64_t prev_t0 = 0;
    int prev_L = 0;
    for (int ch = a; ch < b; ++ch) {
        const int i = ch - a, stage = i % S2_NSTAGE, set = i & 1;
        uint8_t *st = sm + stage * S2_STAGE;
        const int64_t t0 = bos + (int64_t)(ch - cb) * C;
        const int L = (int)((eos - t0) < C ? (eos - t0) : C);
        if (!issuer) {
            // S (fp16) -> B operand [K = dk][N = 32], MN-major, no swizzle:
            // core matrix (8 K rows x 8 N) at (n/8) * 2048 + (k/8) * 128
#pragma unroll
            for (int gq = 0; gq < DVS / 8; ++gq) {
                uint4 v4 = make_uint4(pack_h2(S[8 * gq + 0], S[8 * gq + 1]), pack_h2(S[8 * gq + 2], S[8 * gq + 3]),
                                      pack_h2(S[8 * gq + 4], S[8 * gq + 5]), pack_h2(S[8 * gq + 6], S[8 * gq + 7]));
                *reinterpret_cast<uint4 *>(sm + S2_SOP + 8192 * set + gq * 2048 + (row >> 3) * 128 +
                                           (row & 7) * 16) = v4;
            }
            fence_async_smem();
        }
        fence_before_sync();
        ok = __syncthreads_and(!bad && mbar_wait(&mbar[stage], (uint32_t)((i / S2_NSTAGE) & 1)));
        fence_after_sync();
        if (!ok) break;

        if (issuer) {                     // round 1
            const uint32_t stb = warp_uniform(smb + (uint32_t)stage * S2_STAGE);
            const uint32_t d_w = warp_uniform(tmem + 128u * (uint32_t)set);
            const uint64_t dwq = sdesc_k_sw128(stb + S2_WQ);
            const uint64_t dso = sdesc(smb + S2_SOP + 8192u * (uint32_t)set, 128, 2048, LAYOUT_NONE);
            if (elect_one()) {
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_f16(d_w, sdesc_add(dwq, (s >> 2) * 16384 + (s & 3) * 32),
                            sdesc_add(dso, 256 * s), id_m64, s > 0);
                mma_commit(&mbar[MB_R1]);
#pragma unroll
                for (int s = 0; s < QS_ROUND1; ++s)   // Q^ rows sit 8 KB after the W rows of each atom
                    mma_f16(d_w + 32, sdesc_add(dwq, 8192 + (s >> 2) * 16384 + (s & 3) * 32),
                            sdesc_add(dso, 256 * s), id_m64, s > 0);
                // chunk i + 2's operands into the stage of chunk i - 1 (a stage
                // not used yet when i = 0): its last reader, chunk i - 1's P U,
                // has completed.  Issued here, where the issuer waits anyway
                // for the U operand, so that they never delay round 2.
                if (ch + 2 < b) {
                    if (i == 0 || mbar_wait(&mbar[MB_R2O + (set ^ 1)], (uint32_t)(((i - 1) >> 1) & 1)))
                        issue_loads(ch + 2, (i + 2) % S2_NSTAGE);
                    else
                        bad = true;
                }
            }
            __syncwarp();
        } else {
            // the first half of the previous chunk's O rows, while W S runs
            if (i > 0 && write_o &&
                !store_o(set ^ 1, prev_t0, prev_L, (uint32_t)(((i - 1) >> 1) & 1), 0))
                bad = true;
            // U = U~ - W S for token row 16 warp + lane (lanes 0-15)
            if (!mbar_wait(&mbar[MB_R1], i & 1)) bad = true;
            fence_after_sync();
            float w0[16], w1[16];
            tmem_ld16(tmem_at(tmem, warp, 128 * set), w0);
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 16), w1);
            tmem_wait_ld();
            const int ur = 16 * warp + (lane & 15);
            float u[DVS];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 x = *reinterpret_cast<const uint4 *>(st + S2_U + u_img_off(ur, q));
                const __half2 *h2 = reinterpret_cast<const __half2 *>(&x);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(h2[e]);
                    const int j = 8 * q + 2 * e;
                    u[j] = u_scale * f.x - (j < 16 ? w0[j] : w1[j - 16]);
                    u[j + 1] = u_scale * f.y - (j + 1 < 16 ? w0[j + 1] : w1[j - 15]);
                }
            }
            if (lane < 16) {
#pragma unroll
                for (int gq = 0; gq < DVS / 8; ++gq) {
                    uint4 v4 = make_uint4(pack_h2(u[8 * gq + 0], u[8 * gq + 1]), pack_h2(u[8 * gq + 2], u[8 * gq + 3]),
                                          pack_h2(u[8 * gq + 4], u[8 * gq + 5]), pack_h2(u[8 * gq + 6], u[8 * gq + 7]));
                    *reinterpret_cast<uint4 *>(sm + S2_UOP + gq * 1024 + (ur >> 3) * 128 + (ur & 7) * 16) = v4;
                }
            }
            fence_async_smem();
        }
        // B2 (all): U is in shared memory.
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (issuer) {                     // round 2, then the loads of chunk i + 2
            const uint32_t stb = warp_uniform(smb + (uint32_t)stage * S2_STAGE);
            const uint32_t d_w = warp_uniform(tmem + 128u * (uint32_t)set);
            const uint64_t dkb = sdesc(stb + S2_KB, 8192, 1024, LAYOUT_SW128);
            const uint64_t dp = sdesc_k_sw128(stb + S2_PZ);
            const uint64_t duo = sdesc(smb + S2_UOP, 128, 1024, LAYOUT_NONE);
            const uint64_t dwq = sdesc_k_sw128(stb + S2_WQ);
            const uint64_t dso = sdesc(smb + S2_SOP + 8192u * (uint32_t)set, 128, 2048, LAYOUT_NONE);
            if (elect_one()) {
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16(d_w + 64, sdesc_add(dkb, 2048 * s), sdesc_add(duo, 256 * s), id_kb, s > 0);
                mma_commit(&mbar[MB_R2S]);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16(d_w + 32, sdesc_add(dp, 32 * s), sdesc_add(duo, 256 * s), id_m64, 1);
#pragma unroll
                for (int s = QS_ROUND1; s < 8; ++s)   // the rest of Q^ S
                    mma_f16(d_w + 32, sdesc_add(dwq, 8192 + (s >> 2) * 16384 + (s & 3) * 32),
                            sdesc_add(dso, 256 * s), id_m64, 1);
                mma_commit(&mbar[MB_R2O + set]);
            }
            __syncwarp();
        } else {
            // the second half, while Kbar^T U runs
            if (i > 0) {
                const uint32_t par = (uint32_t)(((i - 1) >> 1) & 1);
                const bool okp = write_o ? store_o(set ^ 1, prev_t0, prev_L, par, 1)
                                         : mbar_wait(&mbar[MB_R2O + (set ^ 1)], par);
                if (!okp) bad = true;
            }
            // S = Diag(e^gamma_last) S + Kbar^T U
            if (!mbar_wait(&mbar[MB_R2S], i & 1)) bad = true;
            fence_after_sync();
            float d2a[16], d2b[16];
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 64), d2a);
            tmem_ld16(tmem_at(tmem, warp, 128 * set + 80), d2b);
            tmem_wait_ld();
            const float gl = reinterpret_cast<const float *>(st + S2_G)[row];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                S[j] = gl * S[j] + d2a[j];
                S[16 + j] = gl * S[16 + j] + d2b[j];
            }
        }
        prev_t0 = t0;
        prev_L = L;
    }
    ok = ok && __syncthreads_and(!bad);
    // the last chunk's outputs (and, in any case, its P U MMA -- the last MMA
    // issued -- before TMEM is freed)
    if (ok && a < b && !issuer) {
        const int il = b - 1 - a;
        const uint32_t par = (uint32_t)((il >> 1) & 1);
        const bool okp = write_o ? (store_o(il & 1, prev_t0, prev_L, par, 0) &&
                                    store_o(il & 1, prev_t0, prev_L, par, 1))
                                 : mbar_wait(&mbar[MB_R2O + (il & 1)], par);
        if (!okp) bad = true;
    }
    ok = __syncthreads_and(ok && !bad);

    if (!ok) {
        // a bounded wait gave up: record it, and let the copies and MMAs this
        // CTA issued finish (bounded waits) before its shared memory and TMEM
        // are released
        if (tid == 0) {
            ws_fail(ws_hdr, 2);
            for (int s2 = 0; s2 < S2_NSTAGE; ++s2)
                if (iss[s2] >= 0)
                    mbar_wait(&mbar[s2], (uint32_t)((iss[s2] / S2_NSTAGE) & 1), 1u << 20);
        }
        if (issuer) {
            if (elect_one()) {
                mma_commit(&mbar[MB_DRAIN]);
                mbar_wait(&mbar[MB_DRAIN], 0, 1u << 20);
            }
            __syncwarp();
        }
    }
    // final state: S_T, or (segment launch) the segment's map, contribution
    // or end state for the combine step; the last segment writes S_T
    float *dst = nullptr;
    if (!p.nseg || (p.phase == 1 && seg == p.nseg - 1))
        dst = p.S_T + sbase_g;
    else if (p.phase == 0)   // segment 0 ends in its B slot
        dst = smap(p.smaps, p.nseg, h, seg, role == SEG_M ? SMAP_M : SMAP_B) + (int64_t)row * D +
              slice * DVS;
    if (dst && !issuer) {
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
// K2, wide form: one CTA per (sequence, head) carrying all 128 state
// columns, for batches with more chains than the GPU runs at once and for the
// state chain that runs beside the per-chunk kernel.  544 threads: warpgroup
// s (warps 4s..4s+3) owns state columns 32s..32s+31, its thread t (0..127)
// row t (a dk channel) of those columns in fp32 registers; warp 16 issues the
// MMAs and the operand loads.  Every MMA spans the whole state (N = 128), so
// one SM carries a whole head in about the period of one 32-column slice.
// Per chunk i (stage and TMEM set i % 2; D_A = set columns 0-127, D_S = set
// columns 128-255):
//   B1 (all):         S (fp16 operand) written, chunk i's operands landed
//   warp 16:          round 1, D_A = [W ; Q^] S (8 K steps) -> MB_R1; then
//                     chunk i + 1's operands into the stage of chunk i - 1,
//                     once that chunk's P U (its last reader) has completed
//   rows 0-63:        U = U~ - W S, fp16 operand
//   rows 64-127:      the O rows of chunk i - 1
//   B2 (all):         U written
//   warp 16:          round 2, D_S = Kbar^T U (4 K steps) -> MB_R2S, then
//                     D_A += [0 ; P] U (4 K steps) -> MB_R2O
//   all state warps:  S = Diag(e^gamma_last) S + D_S   (after MB_R2S)
__global__ void __launch_bounds__(K2W_THREADS, 1) chain_wide_kernel(const K2Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    // [0..1] loads, [2] round 1, [3] round 2 state part, [4] round 2 output part, [5] drain
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + S2W_MISC);
    constexpr int MB_R1 = 2, MB_R2S = 3, MB_R2O = 4, MB_DRAIN = 5;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mbar + 6);
    int32_t *iss = reinterpret_cast<int32_t *>(tmem_slot + 1);   // [2] last chunk loaded per stage

    const int tid = threadIdx.x, lane = tid & 31;
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);   // warp-uniform for the compiler
    const bool issuer = warp == K2W_ISSUER;
    const int wg = (warp >> 2) & 3, wq = warp & 3;   // column block, TMEM lane quadrant
    const int row = 32 * wq + lane;                   // state row (dk channel) / TMEM lane
    const int col0 = 32 * wg;                         // first state column of this thread
    const int H = p.H;
    const int h = blockIdx.x % H;
    int n = blockIdx.x / H;
    if (p.plan) {   // many sequences: the window plan's order, if it picked this form
        if (p.plan[0] != PLAN_WIDE || (int)blockIdx.x >= p.plan[1] * H) return;
        n = p.plan[2 + blockIdx.x / H];
    }
    int32_t *ws_hdr = reinterpret_cast<int32_t *>(p.ws);
    const int32_t *chunk_base = reinterpret_cast<const int32_t *>(p.ws + WS_HEADER);
    const uint8_t *img_base = p.ws + ws_images_offset(p.N);
    if (*reinterpret_cast<volatile int32_t *>(ws_hdr) != 0) return;   // see chain_kernel

    const int cb = chunk_base[n], ce = chunk_base[n + 1];
    const int a = max(cb, p.w0), b = min(ce, p.w1);
    const int64_t sbase = ((int64_t)n * H + h) * D * D + (int64_t)row * D + col0;
    if (cb == ce) {                       // empty sequence: pass the state through
        if (p.w0 == 0 && !issuer) {
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
            float4 x = (src && !issuer) ? *reinterpret_cast<const float4 *>(src + sbase + j)
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
        for (int j = 0; j <= MB_DRAIN; ++j) mbar_init(&mbar[j], 1);
        mbar_fence_init();
        iss[0] = iss[1] = -1;
    }
    if (warp == 0) tmem_alloc<512>(tmem_slot);
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = warp_uniform(*tmem_slot);
    const uint32_t smb = warp_uniform(smem_addr(sm));

    auto issue_loads = [&](int ch, int stage) {
        const uint8_t *src = img_base + ((uint64_t)(ch - p.img0) * H + h) * CH_STRIDE;
        uint8_t *dst = sm + stage * S2W_STAGE;
        uint64_t *mb = &mbar[stage];
        iss[stage] = ch - a;
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
    if (issuer) {                 // chunks a and a + 1 up front
        if (elect_one()) {
            issue_loads(a, 0);
            if (a + 1 < b) issue_loads(a + 1, 1);
        }
        __syncwarp();
    }

    constexpr uint32_t id_wq = idesc(128, 128, FMT_F16, FMT_F16, 0, 1);
    constexpr uint32_t id_kb = idesc(128, 128, FMT_F16, FMT_F16, 1, 1);

    // the O rows of a finished chunk (rows 64-127), once its P U MMA has completed
    auto store_o = [&](int set, int64_t t0, int L, uint32_t pu_parity) -> bool {
        if (!mbar_wait(&mbar[MB_R2O], pu_parity)) return false;
        fence_after_sync();
        float oa[16], ob[16];
        tmem_ld16(tmem_at(tmem, wq, 256 * set + col0), oa);
        tmem_ld16(tmem_at(tmem, wq, 256 * set + col0 + 16), ob);
        tmem_wait_ld();
        const int r = row - 64;
        if (r < L) {
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
        return true;
    };

    bool ok = true, bad = false;
    int64_t prev_t0 = 0;
    int prev_L = 0;
    for (int ch = a; ch < b; ++ch) {
        const int i = ch - a, stage = i & 1, set = i & 1;
        uint8_t *st = sm + stage * S2W_STAGE;
        const int64_t t0 = bos + (int64_t)(ch - cb) * C;
        const int L = (int)((eos - t0) < C ? (eos - t0) : C);
        if (!issuer) {
            // S (fp16) -> B operand [K = dk][N = 128], MN-major, 128-byte
            // swizzle: two 64-column atoms of 128 rows x 128 bytes
#pragma unroll
            for (int gq = 0; gq < 4; ++gq) {
                uint4 v4 = make_uint4(pack_h2(S[8 * gq + 0], S[8 * gq + 1]), pack_h2(S[8 * gq + 2], S[8 * gq + 3]),
                                      pack_h2(S[8 * gq + 4], S[8 * gq + 5]), pack_h2(S[8 * gq + 6], S[8 * gq + 7]));
                *reinterpret_cast<uint4 *>(sm + S2W_SOP + (wg >> 1) * 16384 +
                                           sw128_off(row, (wg & 1) * 4 + gq)) = v4;
            }
            fence_async_smem();
        }
        fence_before_sync();
        ok = __syncthreads_and(!bad && mbar_wait(&mbar[stage], (uint32_t)((i >> 1) & 1)));
        fence_after_sync();
        if (!ok) break;

        if (issuer) {                     // round 1, then the loads of chunk i + 1
            const uint32_t stb = warp_uniform(smb + (uint32_t)stage * S2W_STAGE);
            const uint32_t d_a = warp_uniform(tmem + 256u * (uint32_t)set);
            const uint64_t dwq = sdesc_k_sw128(stb + S2W_WQ);
            const uint64_t dso = sdesc(smb + S2W_SOP, 16384, 1024, LAYOUT_SW128);
            if (elect_one()) {
#pragma unroll
                for (int s8 = 0; s8 < 8; ++s8)
                    mma_f16(d_a, sdesc_add(dwq, (s8 >> 2) * 16384 + (s8 & 3) * 32),
                            sdesc_add(dso, 2048 * s8), id_wq, s8 > 0);
                mma_commit(&mbar[MB_R1]);
                if (i > 0 && ch + 1 < b) {
                    if (mbar_wait(&mbar[MB_R2O], (uint32_t)((i - 1) & 1)))
                        issue_loads(ch + 1, stage ^ 1);
                    else
                        bad = true;
                }
            }
            __syncwarp();
        } else if (wq < 2) {              // U = U~ - W S for token rows 0-63
            if (!mbar_wait(&mbar[MB_R1], i & 1)) bad = true;
            fence_after_sync();
            float w0[16], w1[16];
            tmem_ld16(tmem_at(tmem, wq, 256 * set + col0), w0);
            tmem_ld16(tmem_at(tmem, wq, 256 * set + col0 + 16), w1);
            tmem_wait_ld();
            float u[32];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const uint4 x = *reinterpret_cast<const uint4 *>(st + S2W_U + wg * 4096 + u_img_off(row, q4));
                const __half2 *h2 = reinterpret_cast<const __half2 *>(&x);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(h2[e]);
                    const int j = 8 * q4 + 2 * e;
                    u[j] = f.x - (j < 16 ? w0[j] : w1[j - 16]);
                    u[j + 1] = f.y - (j + 1 < 16 ? w0[j + 1] : w1[j - 15]);
                }
            }
#pragma unroll
            for (int gq = 0; gq < 4; ++gq) {
                uint4 v4 = make_uint4(pack_h2(u[8 * gq + 0], u[8 * gq + 1]), pack_h2(u[8 * gq + 2], u[8 * gq + 3]),
                                      pack_h2(u[8 * gq + 4], u[8 * gq + 5]), pack_h2(u[8 * gq + 6], u[8 * gq + 7]));
                *reinterpret_cast<uint4 *>(sm + S2W_UOP + (wg >> 1) * 8192 +
                                           sw128_off(row, (wg & 1) * 4 + gq)) = v4;
            }
            fence_async_smem();
        } else if (i > 0) {               // rows 64-127: the previous chunk's outputs
            if (!store_o(set ^ 1, prev_t0, prev_L, (uint32_t)((i - 1) & 1))) bad = true;
        }
        // B2 (all): U is in shared memory; every thread has seen chunk i - 1's
        // P U complete before the issuer commits chunk i's
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (issuer) {                     // round 2
            const uint32_t stb = warp_uniform(smb + (uint32_t)stage * S2W_STAGE);
            const uint32_t d_a = warp_uniform(tmem + 256u * (uint32_t)set);
            const uint64_t dkb = sdesc(stb + S2W_KB, 8192, 1024, LAYOUT_SW128);
            const uint64_t dpz = sdesc_k_sw128(stb + S2W_PZ);
            const uint64_t duo = sdesc(smb + S2W_UOP, 8192, 1024, LAYOUT_SW128);
            if (elect_one()) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16(d_a + 128, sdesc_add(dkb, 2048 * ks), sdesc_add(duo, 2048 * ks), id_kb, ks > 0);
                mma_commit(&mbar[MB_R2S]);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16(d_a, sdesc_add(dpz, 32 * ks), sdesc_add(duo, 2048 * ks), id_wq, 1);
                mma_commit(&mbar[MB_R2O]);
            }
            __syncwarp();
        } else {                          // S = Diag(e^gamma_last) S + Kbar^T U
            if (!mbar_wait(&mbar[MB_R2S], i & 1)) bad = true;
            fence_after_sync();
            float da[16], db[16];
            tmem_ld16(tmem_at(tmem, wq, 256 * set + 128 + col0), da);
            tmem_ld16(tmem_at(tmem, wq, 256 * set + 128 + col0 + 16), db);
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
    }
    ok = ok && __syncthreads_and(!bad);
    // the last chunk's outputs (its P U is the last MMA issued, so TMEM is
    // idle afterwards)
    if (ok && !issuer && wq >= 2) {
        if (!store_o((b - 1 - a) & 1, prev_t0, prev_L, (uint32_t)((b - 1 - a) & 1))) bad = true;
    }
    ok = __syncthreads_and(ok && !bad);

    if (!ok) {
        // a bounded wait gave up: record it, and let the copies and MMAs this
        // CTA issued finish (bounded waits) before its shared memory and TMEM
        // are released
        if (tid == 0) {
            ws_fail(ws_hdr, 2);
            for (int s2 = 0; s2 < 2; ++s2)
                if (iss[s2] >= 0) mbar_wait(&mbar[s2], (uint32_t)((iss[s2] >> 1) & 1), 1u << 20);
        }
        if (issuer) {
            if (elect_one()) {
                mma_commit(&mbar[MB_DRAIN]);
                mbar_wait(&mbar[MB_DRAIN], 0, 1u << 20);
            }
            __syncwarp();
        }
    }
    if (!issuer) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4 *>(p.S_T + sbase + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc<512>(tmem);
}

}  // namespace tcp
}  // namespace kda
