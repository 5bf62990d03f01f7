// kda_decode.cu -- batched KDA decode step (one token per sequence).
//
// Per (sequence, head), with the fp32 state S [D x D] updated in place:
//   S' = Diag(exp g) S;  w = S'^T k;  u = beta (v - w);  S = S' + k u^T;
//   o  = S^T q = S'^T q + (q . k) u
// (decay first, read the stored value, write only the delta: the lineage
// essay "GPT-2부터 Kimi K3까지", sections "DeltaNet" and "Gated DeltaNet";
// per-channel gate: its section "KDA: Kimi의 비법").
//
// Decode is bound by HBM bandwidth (the essay's section "KV 캐시: 재계산하지
// 말고 저장하라" makes the same point for the KV cache this state replaces):
// the state is 64 KB per head at D = 128 and every step must read and write
// all of it, while the per-token vectors are < 1.5 KB.  So one CTA owns one
// (sequence, head), issues all of its state loads up front as coalesced
// 128-bit streaming loads (each warp instruction covers one 512-byte row),
// keeps the state in registers, reduces S'^T k and S'^T q across the CTA and
// writes the updated state back once with 128-bit streaming stores.  Nothing
// but the state touches HBM in bulk.
#include "kda_internal.cuh"

namespace kda {
namespace {

template <int D, int ROWS>
struct DecodeShape {
    static constexpr int LANES = D / 4;          // float4 columns per row
    static constexpr int GROUPS = D / ROWS;      // row groups
    static constexpr int NT = GROUPS * LANES;    // threads per CTA
};

// POOLED: the state of sequence b lives in slot slots[b] of a pool of P
// states [P, H, D, D]; a slot outside [0, P) skips the sequence (its o row is
// zeroed and no state is touched).
template <int D, int ROWS, typename Tin, bool POOLED>
__global__ void __launch_bounds__(DecodeShape<D, ROWS>::NT)
decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
              const Tin *__restrict__ v, const float *__restrict__ g,
              const float *__restrict__ beta, float *__restrict__ S,
              Tin *__restrict__ o, const int32_t *__restrict__ slots, int H, int P,
              bool scalar_gate) {
    using Sh = DecodeShape<D, ROWS>;
    constexpr int LANES = Sh::LANES, GROUPS = Sh::GROUPS, NT = Sh::NT;
    // Launched as a programmatic dependent: the CTAs may become resident while
    // the previous kernel on the stream (typically the previous decode step,
    // which writes these states) is still finishing; every global access
    // comes after the wait for its completion.  Once every CTA of this step
    // has started, the next step may be launched the same way.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    const int lane = tid % LANES;
    const int grp = tid / LANES;
    const int64_t bh = blockIdx.x;               // sequence * H + head
    int64_t sidx = bh;                           // which state
    if (POOLED) {
        const int slot = slots[bh / H];
        if (slot < 0 || slot >= P) {
            for (int i = tid; i < LANES; i += NT)
                store4(o + bh * D + 4 * i, make_float4(0.f, 0.f, 0.f, 0.f));
            return;
        }
        sidx = (int64_t)slot * H + bh % H;
    }

    float4 *Sp = reinterpret_cast<float4 *>(S + sidx * (int64_t)D * D);
    float4 s[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
        s[r] = __ldcs(Sp + (grp * ROWS + r) * LANES + lane);

    __shared__ float sk[D], sq[D], sa[D];
    __shared__ float4 sv4[LANES], su4[LANES];
    __shared__ float4 red_w[GROUPS][LANES], red_z[GROUPS][LANES];
    __shared__ float sqk;

    const int64_t vb = bh * D;
    for (int i = tid; i < D; i += NT) {
        sk[i] = to_f32(k[vb + i]);
        sq[i] = to_f32(q[vb + i]);
        sa[i] = expf(scalar_gate ? g[bh] : g[vb + i]);
    }
    for (int i = tid; i < LANES; i += NT)
        sv4[i] = load4(v + vb + 4 * i);
    const float b = beta[bh];
    __syncthreads();

    float4 pw = make_float4(0.f, 0.f, 0.f, 0.f), pz = pw;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const int row = grp * ROWS + r;
        const float a = sa[row], kr = sk[row], qr = sq[row];
        s[r].x *= a; s[r].y *= a; s[r].z *= a; s[r].w *= a;
        pw.x += s[r].x * kr; pw.y += s[r].y * kr; pw.z += s[r].z * kr; pw.w += s[r].w * kr;
        pz.x += s[r].x * qr; pz.y += s[r].y * qr; pz.z += s[r].z * qr; pz.w += s[r].w * qr;
    }
    red_w[grp][lane] = pw;
    red_z[grp][lane] = pz;
    if (tid < 32) {                              // q . k on one warp
        float acc = 0.f;
        for (int i = tid; i < D; i += 32) acc += sq[i] * sk[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (tid == 0) sqk = acc;
    }
    __syncthreads();

    if (tid < LANES) {
        float4 w = red_w[0][tid], z = red_z[0][tid];
#pragma unroll
        for (int gi = 1; gi < GROUPS; ++gi) {
            const float4 a = red_w[gi][tid], c = red_z[gi][tid];
            w.x += a.x; w.y += a.y; w.z += a.z; w.w += a.w;
            z.x += c.x; z.y += c.y; z.z += c.z; z.w += c.w;
        }
        const float4 vv = sv4[tid];
        float4 u;
        u.x = b * (vv.x - w.x); u.y = b * (vv.y - w.y);
        u.z = b * (vv.z - w.z); u.w = b * (vv.w - w.w);
        const float qk = sqk;
        float4 out;
        out.x = z.x + qk * u.x; out.y = z.y + qk * u.y;
        out.z = z.z + qk * u.z; out.w = z.w + qk * u.w;
        store4(o + vb + 4 * tid, out);
        su4[tid] = u;
    }
    __syncthreads();

    const float4 u = su4[lane];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const float kr = sk[grp * ROWS + r];
        s[r].x += kr * u.x; s[r].y += kr * u.y; s[r].z += kr * u.z; s[r].w += kr * u.w;
        __stcs(Sp + (grp * ROWS + r) * LANES + lane, s[r]);
    }
}

// Consecutive decode steps are separate launches of ~160 us each (1 GiB of
// state at B = 256, H = 32); launching each as a programmatic dependent of the
// previous kernel hides the launch and CTA ramp-up (~2 us per step measured
// between back-to-back launches) behind the previous step's last wave.
template <int D, int ROWS, typename Tin, bool POOLED>
cudaError_t launch(const DecodeArgs &a, cudaStream_t st) {
    const int64_t units = (int64_t)a.B * a.H;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)units);
    cfg.blockDim = dim3(DecodeShape<D, ROWS>::NT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_kernel<D, ROWS, Tin, POOLED>, (const Tin *)a.q,
                              (const Tin *)a.k, (const Tin *)a.v, a.g, a.beta, a.S, (Tin *)a.o,
                              a.slots, a.H, a.P, a.scalar_gate);
}

template <bool POOLED>
cudaError_t dispatch(const DecodeArgs &a, cudaStream_t st) {
    if ((int64_t)a.B * a.H == 0) return cudaSuccess;
    const bool bf = a.dtype == 0;
    if (a.dk == 128)
        return bf ? launch<128, 16, __nv_bfloat16, POOLED>(a, st) : launch<128, 16, float, POOLED>(a, st);
    return bf ? launch<64, 16, __nv_bfloat16, POOLED>(a, st) : launch<64, 16, float, POOLED>(a, st);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st) {
    return a.slots ? dispatch<true>(a, st) : dispatch<false>(a, st);
}

}  // namespace kda
