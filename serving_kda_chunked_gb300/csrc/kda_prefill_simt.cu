// kda_prefill_simt.cu -- chunked KDA prefill on CUDA cores, fp32 arithmetic.
//
// This is the fp32 path (fp32 q/k/v/o) and the arithmetic scaffold of the
// tensor-core path: it runs the same chunked algebra with every product in
// fp32 on CUDA cores.
//
// Chunking follows the lineage essay "GPT-2부터 Kimi K3까지", section
// "병렬화 트릭": within a chunk of C = 64 tokens the deltas are resolved all
// at once (a unit-lower-triangular solve, the UT form of the Householder
// reparameterisation), and only the state crosses chunk boundaries.  For the
// per-channel gate (section "KDA: Kimi의 비법") and a chunk entering with
// state S, with gamma = per-channel cumulative log-gate inside the chunk:
//
//   A[r,i] = beta_r sum_c k_rc k_ic exp(gamma_rc - gamma_ic)   (i < r)
//   P[r,i] =        sum_c q_rc k_ic exp(gamma_rc - gamma_ic)   (i <= r)
//   (I + A) U = Diag(beta) (V - (K * exp(gamma)) S)
//   O      = (Q * exp(gamma)) S + P U
//   S_next = Diag(exp(gamma_last)) S + (K * exp(gamma_last - gamma))^T U
//
// While no channel decays below e^-80 over the chunk, the pair factor is
// split as exp(gamma_rc) * exp(-gamma_ic), both inside fp32, and A and P are
// plain products of the scaled rows (2 exponentials per element instead of
// one per pair and channel).  Otherwise each pair's exponent is formed first;
// it is <= 0 (pairs with i <= r only), so nothing can overflow.  Columns of S
// are independent, so one CTA owns one (sequence, head, block of DVS state
// columns) and walks the sequence's chunks in order with its state slice in
// shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int C = 64;      // tokens per chunk
constexpr int NT = 256;    // threads per CTA
constexpr float RANGE_LIMIT = 80.f;   // e^80 stays inside fp32

template <int DK, int DVS>
struct SimtSmem {
    static constexpr int KP = DK + 1;  // padded row stride of [C][DK] tiles
    static constexpr int CP = C + 1;   // padded row stride of [C][C] tiles
    static constexpr size_t floats =
        4 * (size_t)C * KP + 2 * (size_t)C * CP + (size_t)DK * DVS +
        (size_t)C * DVS + C + 2 * DK + NT;
    static constexpr size_t bytes = floats * sizeof(float);
};

template <int DK, int DVS, typename Tin>
__global__ void __launch_bounds__(NT, 1)
prefill_simt_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                    const Tin *__restrict__ v, const float *__restrict__ g,
                    const float *__restrict__ beta, const float *S0,
                    const int32_t *__restrict__ cu, Tin *__restrict__ o,
                    float *S_T, int H, int64_t T, int n_slices, bool scalar_gate) {
    using Sm = SimtSmem<DK, DVS>;
    constexpr int KP = Sm::KP, CP = Sm::CP;
    constexpr int DV = DK;
    extern __shared__ float smem[];
    float *sK = smem;              // [C][KP]  k, then k * exp(gamma)
    float *sQ = sK + C * KP;       // [C][KP]  q, then q * exp(gamma)
    float *sG = sQ + C * KP;       // [C][KP]  g, then gamma, then kbar
    float *sKn = sG + C * KP;      // [C][KP]  k * exp(-gamma) (single-reference chunks)
    float *sA = sKn + C * KP;      // [C][CP]  A
    float *sP = sA + C * CP;       // [C][CP]  P
    float *sS = sP + C * CP;       // [DK][DVS] state slice
    float *sV = sS + DK * DVS;     // [C][DVS] v, then rhs, then U
    float *sB = sV + C * DVS;      // [C] beta
    float *sGL = sB + C;           // [DK] gamma at the chunk's last row
    float *sEL = sGL + DK;         // [DK] exp(gamma_last)
    float *sTot = sEL + DK;        // [NT / DK][DK] per-segment gate sums

    const int tid = threadIdx.x;
    const int unit = blockIdx.x;
    const int slice = unit % n_slices;
    const int h = (unit / n_slices) % H;
    const int n = unit / (n_slices * H);
    const int col0 = slice * DVS;
    int64_t bos, eos;
    seq_bounds(cu, n, T, bos, eos);

    const int64_t sbase = ((int64_t)n * H + h) * DK * DV;
    for (int idx = tid; idx < DK * DVS; idx += NT) {
        const int c = idx / DVS, j = idx % DVS;
        sS[idx] = S0 ? S0[sbase + (int64_t)c * DV + col0 + j] : 0.f;
    }

    for (int64_t c0 = bos; c0 < eos; c0 += C) {
        const int L = (int)((eos - c0) < C ? (eos - c0) : C);
        // ---- stage the chunk; rows past the sequence end are no-op tokens
        // (four rows' loads in flight per thread before any is stored)
        static_assert((C * DK) % (4 * NT) == 0, "staging in rounds of four");
        for (int idx0 = tid; idx0 < C * DK; idx0 += 4 * NT) {
            float kv[4], qv[4], gv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int idx = idx0 + u * NT, r = idx / DK, c = idx % DK;
                kv[u] = qv[u] = gv[u] = 0.f;
                if (r < L) {
                    const int64_t off = ((c0 + r) * H + h) * DK + c;
                    kv[u] = to_f32(k[off]);
                    qv[u] = to_f32(q[off]);
                    gv[u] = scalar_gate ? g[(c0 + r) * H + h] : g[off];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int idx = idx0 + u * NT, r = idx / DK, c = idx % DK;
                sK[r * KP + c] = kv[u];
                sQ[r * KP + c] = qv[u];
                sG[r * KP + c] = gv[u];
            }
        }
        for (int idx = tid; idx < C * DVS; idx += NT) {
            const int r = idx / DVS, j = idx % DVS;
            sV[idx] = r < L ? to_f32(v[((c0 + r) * H + h) * DV + col0 + j]) : 0.f;
        }
        for (int r = tid; r < C; r += NT)
            sB[r] = r < L ? beta[(c0 + r) * H + h] : 0.f;
        __syncthreads();

        // ---- per-channel cumulative log-gate: thread (channel c, row segment
        // sg) scans its segment, then adds the totals of the segments before it
        {
            constexpr int NSEG = NT / DK, SEG = C / NSEG;
            static_assert(NT % DK == 0 && C % NSEG == 0, "row segments");
            const int c = tid % DK, sg = tid / DK;
            float acc = 0.f;
#pragma unroll 4
            for (int r = sg * SEG; r < (sg + 1) * SEG; ++r) {
                acc += sG[r * KP + c];
                sG[r * KP + c] = acc;
            }
            sTot[sg * DK + c] = acc;
            __syncthreads();
            float off = 0.f;
            for (int s2 = 0; s2 < sg; ++s2) off += sTot[s2 * DK + c];
            if (sg > 0) {
#pragma unroll 4
                for (int r = sg * SEG; r < (sg + 1) * SEG; ++r) sG[r * KP + c] += off;
            }
            if (sg == NSEG - 1) {
                sGL[c] = acc + off;
                sEL[c] = expf(acc + off);
            }
        }
        __syncthreads();

        const bool single_ref = __syncthreads_and(tid >= DK || sGL[tid] >= -RANGE_LIMIT);
        if (single_ref) {
            // ---- K*exp(gamma), Q*exp(gamma), K*exp(-gamma) and
            // kbar = K*exp(-gamma)*exp(gamma_last)
            for (int idx = tid; idx < C * DK; idx += NT) {
                const int r = idx / DK, c = idx % DK;
                const float gam = sG[r * KP + c];
                const float kk = sK[r * KP + c];
                const float kn = kk * expf(-gam);
                const float e = expf(gam);
                sKn[r * KP + c] = kn;
                sG[r * KP + c] = kn * sEL[c];
                sK[r * KP + c] = kk * e;
                sQ[r * KP + c] *= e;
            }
            __syncthreads();
            // ---- gated K K^T (strictly lower, times beta_r) and Q K^T (lower):
            // thread t owns rows 4 (t / 16) + u and columns t % 16 + 16 w
            // (u, w < 4), so that a warp's column loads hit 16 distinct banks
            static_assert(NT == 256 && C == 64, "one 4 x 4 tile of the 64 x 64 products per thread");
            {
                const int r0 = 4 * (tid >> 4), i0 = tid & 15;
                float a[4][4] = {}, pq[4][4] = {};
                const float *kr = sK + r0 * KP, *qr = sQ + r0 * KP, *ki = sKn + i0 * KP;
#pragma unroll 4
                for (int c = 0; c < DK; ++c) {
                    float x[4], y[4], z[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        x[u] = kr[u * KP + c];
                        y[u] = qr[u * KP + c];
                        z[u] = ki[16 * u * KP + c];
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            a[u][w] = fmaf(x[u], z[w], a[u][w]);
                            pq[u][w] = fmaf(y[u], z[w], pq[u][w]);
                        }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int r = r0 + u, i = i0 + 16 * w;
                        sA[r * CP + i] = i < r ? sB[r] * a[u][w] : 0.f;
                        sP[r * CP + i] = i <= r ? pq[u][w] : 0.f;
                    }
            }
        } else {
            // ---- the same with each pair's exponent formed first
            for (int pidx = tid; pidx < C * C; pidx += NT) {
                const int r = pidx / C, i = pidx % C;
                float a = 0.f, p = 0.f;
                if (i <= r) {
                    const float *gr = sG + r * KP, *gi = sG + i * KP;
                    const float *kr = sK + r * KP, *ki = sK + i * KP, *qr = sQ + r * KP;
#pragma unroll 4
                    for (int c = 0; c < DK; ++c) {
                        const float kie = ki[c] * expf(gr[c] - gi[c]);
                        a += kr[c] * kie;
                        p += qr[c] * kie;
                    }
                }
                sA[r * CP + i] = i < r ? sB[r] * a : 0.f;
                sP[r * CP + i] = p;
            }
            __syncthreads();
            for (int idx = tid; idx < C * DK; idx += NT) {
                const int r = idx / DK, c = idx % DK;
                const float gam = sG[r * KP + c];
                const float e = expf(gam);
                const float kk = sK[r * KP + c];
                sG[r * KP + c] = kk * expf(sGL[c] - gam);
                sK[r * KP + c] = kk * e;
                sQ[r * KP + c] *= e;
            }
        }
        __syncthreads();

        // [C][DVS] results below: thread t owns rows r2, r2 + 1 and columns
        // j4 .. j4 + 3 (state rows are read as float4)
        static_assert(C * DVS == 8 * NT, "two rows x four columns per thread");
        const int j4 = 4 * (tid % (DVS / 4)), r2 = 2 * (tid / (DVS / 4));

        // ---- right-hand side: beta (V - (K*exp(gamma)) S)
        {
            float acc[2][4] = {};
            const float *k0 = sK + r2 * KP;
#pragma unroll 4
            for (int c = 0; c < DK; ++c) {
                const float4 s4 = *reinterpret_cast<const float4 *>(sS + c * DVS + j4);
                const float x0 = k0[c], x1 = k0[KP + c];
                acc[0][0] = fmaf(x0, s4.x, acc[0][0]); acc[0][1] = fmaf(x0, s4.y, acc[0][1]);
                acc[0][2] = fmaf(x0, s4.z, acc[0][2]); acc[0][3] = fmaf(x0, s4.w, acc[0][3]);
                acc[1][0] = fmaf(x1, s4.x, acc[1][0]); acc[1][1] = fmaf(x1, s4.y, acc[1][1]);
                acc[1][2] = fmaf(x1, s4.z, acc[1][2]); acc[1][3] = fmaf(x1, s4.w, acc[1][3]);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float *vr = sV + (r2 + u) * DVS + j4;
                const float b = sB[r2 + u];
#pragma unroll
                for (int w = 0; w < 4; ++w) vr[w] = b * (vr[w] - acc[u][w]);
            }
        }
        __syncthreads();

        // ---- forward substitution (I + A) U = rhs; warp w solves columns
        // w, w + 8, ... together (independent chains, one load of A per row)
        {
            constexpr int NW = NT / 32, CPW = DVS / NW;
            static_assert(DVS % NW == 0, "columns per warp");
            const int warp = tid / 32, lane = tid % 32;
            float x0[CPW], x1[CPW];
#pragma unroll
            for (int m = 0; m < CPW; ++m) {
                x0[m] = sV[lane * DVS + warp + NW * m];
                x1[m] = sV[(lane + 32) * DVS + warp + NW * m];
            }
            for (int r = 0; r < C; ++r) {
                const float a0 = sA[lane * CP + r], a1 = sA[(lane + 32) * CP + r];
#pragma unroll
                for (int m = 0; m < CPW; ++m) {
                    const float ur = __shfl_sync(0xffffffffu, r < 32 ? x0[m] : x1[m], r & 31);
                    if (lane > r) x0[m] -= a0 * ur;
                    if (lane + 32 > r) x1[m] -= a1 * ur;
                }
            }
#pragma unroll
            for (int m = 0; m < CPW; ++m) {
                sV[lane * DVS + warp + NW * m] = x0[m];
                sV[(lane + 32) * DVS + warp + NW * m] = x1[m];
            }
        }
        __syncthreads();

        // ---- outputs O = (Q*exp(gamma)) S + P U (P is zero above the diagonal)
        {
            float acc[2][4] = {};
            const float *q0 = sQ + r2 * KP;
#pragma unroll 4
            for (int c = 0; c < DK; ++c) {
                const float4 s4 = *reinterpret_cast<const float4 *>(sS + c * DVS + j4);
                const float x0 = q0[c], x1 = q0[KP + c];
                acc[0][0] = fmaf(x0, s4.x, acc[0][0]); acc[0][1] = fmaf(x0, s4.y, acc[0][1]);
                acc[0][2] = fmaf(x0, s4.z, acc[0][2]); acc[0][3] = fmaf(x0, s4.w, acc[0][3]);
                acc[1][0] = fmaf(x1, s4.x, acc[1][0]); acc[1][1] = fmaf(x1, s4.y, acc[1][1]);
                acc[1][2] = fmaf(x1, s4.z, acc[1][2]); acc[1][3] = fmaf(x1, s4.w, acc[1][3]);
            }
            const float *p0 = sP + r2 * CP;
            for (int i = 0; i <= r2 + 1; ++i) {
                const float4 u4 = *reinterpret_cast<const float4 *>(sV + i * DVS + j4);
                const float x0 = p0[i], x1 = p0[CP + i];
                acc[0][0] = fmaf(x0, u4.x, acc[0][0]); acc[0][1] = fmaf(x0, u4.y, acc[0][1]);
                acc[0][2] = fmaf(x0, u4.z, acc[0][2]); acc[0][3] = fmaf(x0, u4.w, acc[0][3]);
                acc[1][0] = fmaf(x1, u4.x, acc[1][0]); acc[1][1] = fmaf(x1, u4.y, acc[1][1]);
                acc[1][2] = fmaf(x1, u4.z, acc[1][2]); acc[1][3] = fmaf(x1, u4.w, acc[1][3]);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (r2 + u < L)
                    store4(o + ((c0 + r2 + u) * H + h) * DV + col0 + j4,
                           make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]));
        }
        __syncthreads();

        // ---- state carry S = Diag(exp(gamma_last)) S + kbar^T U: thread t
        // owns state rows c2, c2 + 1 (+ 64 per pass) and columns j4 .. j4 + 3
#pragma unroll
        for (int pass = 0; pass < DK / 64; ++pass) {
            const int c2 = 64 * pass + r2;
            float acc[2][4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float4 s4 = *reinterpret_cast<const float4 *>(sS + (c2 + u) * DVS + j4);
                const float e = sEL[c2 + u];
                acc[u][0] = e * s4.x; acc[u][1] = e * s4.y; acc[u][2] = e * s4.z; acc[u][3] = e * s4.w;
            }
#pragma unroll 4
            for (int r = 0; r < C; ++r) {
                const float4 u4 = *reinterpret_cast<const float4 *>(sV + r * DVS + j4);
                const float x0 = sG[r * KP + c2], x1 = sG[r * KP + c2 + 1];
                acc[0][0] = fmaf(x0, u4.x, acc[0][0]); acc[0][1] = fmaf(x0, u4.y, acc[0][1]);
                acc[0][2] = fmaf(x0, u4.z, acc[0][2]); acc[0][3] = fmaf(x0, u4.w, acc[0][3]);
                acc[1][0] = fmaf(x1, u4.x, acc[1][0]); acc[1][1] = fmaf(x1, u4.y, acc[1][1]);
                acc[1][2] = fmaf(x1, u4.z, acc[1][2]); acc[1][3] = fmaf(x1, u4.w, acc[1][3]);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u)   // rows only this thread reads
                *reinterpret_cast<float4 *>(sS + (c2 + u) * DVS + j4) =
                    make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
        }
        __syncthreads();
    }

    for (int idx = tid; idx < DK * DVS; idx += NT) {
        const int c = idx / DVS, j = idx % DVS;
        S_T[sbase + (int64_t)c * DV + col0 + j] = sS[idx];
    }
}

template <int DK, int DVS, typename Tin>
cudaError_t launch(const PrefillArgs &a, cudaStream_t st) {
    using Sm = SimtSmem<DK, DVS>;
    auto kern = prefill_simt_kernel<DK, DVS, Tin>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Sm::bytes);
    if (e != cudaSuccess) return e;
    const int n_slices = DK / DVS;
    const int64_t units = (int64_t)a.N * a.H * n_slices;
    kern<<<(unsigned)units, NT, Sm::bytes, st>>>(
        (const Tin *)a.q, (const Tin *)a.k, (const Tin *)a.v, a.g, a.beta, a.S0,
        a.cu_seqlens, (Tin *)a.o, a.S_T, a.H, a.T, n_slices, a.scalar_gate);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs &a, cudaStream_t st) {
    if ((int64_t)a.N * a.H == 0) return cudaSuccess;
    const bool bf = a.dtype == 0;
    if (a.dk == 128)
        return bf ? launch<128, 32, __nv_bfloat16>(a, st) : launch<128, 32, float>(a, st);
    return bf ? launch<64, 32, __nv_bfloat16>(a, st) : launch<64, 32, float>(a, st);
}

}  // namespace kda
