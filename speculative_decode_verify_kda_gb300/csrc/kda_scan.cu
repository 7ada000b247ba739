// kda_scan.cu -- the fused KDA verify walk (short conv, activations, gated delta
// rule) for sm_103a, and the accept-j rollback that replays it.
//
// Work decomposition.  One CTA owns one (layer, session, head) unit: 128 threads,
// each holding a 64-row x 2-column tile of the head's 128 x 128 f32 state in
// registers for the whole T-row loop, so the 64 KiB state of a head crosses HBM
// once in and once out per round (plus the fused snapshot write).  Thread
// (warp w, lane L) owns columns j0 = 32w + 2*(L>>1) and j0+1 and key rows
// i = 8g + 4*(L&1) + r (g < 16, r < 4); row pairs (i, i+1) of one column are
// packed into a float2 so the per-row work runs on the packed f32x2 pipe
// (__fmul2_rn / __ffma2_rn).  The two lanes L, L^1 that share a column pair
// finish the reductions over i with one shuffle each.
//
// Per row t (glm_spec.rs module doc, VERIFY-ROW BATCHING: the recurrence stays
// sequential inside one launch, the in-kernel T-loop being the chained t=1
// program):
//   S' = d_t (.) S               d = exp(g), g = -5 sigmoid(raw_g)
//   u  = S'^T k,  e = S'^T q     one register sweep
//   w  = beta (v - u)
//   o  = (e + w (k.q)) / sqrt(128)   == (S' + k w^T)^T q / sqrt(128)
//   S  = S' + k w^T              second register sweep
// Every operation is an explicitly rounded intrinsic and the code for a row does
// not depend on T, so T rows in one launch and T launches of one row give the
// same bits.
//
// Prologue per CTA: the raw rows of the unit (and the 3-slot conv ring) are
// widened into shared memory; one warp per row then computes the width-4 causal
// conv + SiLU of q, k, v (mini fixture linear_attn_config of
// glm5_spec_ppn_gate.rs: short_conv_kernel_size 4, head_dim 128,
// gate_lower_bound -5.0), the L2 norms of q and k, k.q, the gates and beta, with
// one fixed reduction tree per row.  The state loads are issued before the
// prologue so their latency hides behind it.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int D = 128;
constexpr int NW = 4;           // warps per CTA
constexpr int NT = NW * 32;     // threads per CTA
constexpr float L2_EPS = 1e-6f;
constexpr float GATE_LOWER_BOUND = -5.0f;
constexpr float OUT_SCALE = 0.0883883476483184405501f;  // 1 / sqrt(128)

enum KeepMode { KEEP_NONE = 0, KEEP_HOST = 1, KEEP_DEVICE = 2 };

struct ScanParams {
    const float *s_in;   // [L][B][H][D][D]
    float *s_out;
    float *s_snap;       // nullable: receives s_in of each unit
    const float *ring_in;  // [L][B][H][3][3][D]
    float *ring_out;
    float *ring_snap;    // nullable: receives ring_in of each unit
    const float *conv_w; // [L][H][3][D][4]
    const void *xq, *xk, *xv, *xg, *xb;  // [L][B][T_rows][H][D], xb [L][B][T_rows][H]
    float *out;          // nullable: [L][B][T_rows][H][D]
    const int *keep_dev; // KEEP_DEVICE: [B]
    int *status;         // nullable device status word
    int L, B, H;
    int T_rows;          // row count of the raw-row tensors
    int T_run;           // rows to run for KEEP_NONE
    int bf16;
    int keep_mode;
    unsigned char keep_host[KDA_HOST_KEEP_MAX];
};

// shared memory for a launch whose units run at most tcap rows
__host__ __device__ constexpr size_t smem_floats(int tcap)
{
    return (size_t)3 * (tcap + 3) * D   // ext: [3 stream][ring slots + rows][D]
           + (size_t)3 * D * 4          // conv weights [3][D] float4
           + (size_t)tcap * 4 * D       // per-row vectors d, k_hat, q_hat, v
           + (size_t)tcap * 2 + 2;      // per-row beta, k.q (+ pad to 16 B)
}

__device__ __forceinline__ float sigmoidf_(float z)
{
    return __frcp_rn(__fadd_rn(1.0f, expf(-z)));
}

__device__ __forceinline__ float bf16_widen(uint16_t b)
{
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float load_scalar(const void *base, int bf16, size_t idx)
{
    if (bf16)
        return bf16_widen(static_cast<const uint16_t *>(base)[idx]);
    return static_cast<const float *>(base)[idx];
}

// butterfly all-reduce over the warp; every lane ends with the same bits
__device__ __forceinline__ float warp_allsum(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}

__device__ __forceinline__ float conv4(float4 w, float x0, float x1, float x2, float x3)
{
    // w.x multiplies x[t-3] (x0), w.w the current row x[t] (x3)
    return __fmaf_rn(w.w, x3, __fmaf_rn(w.z, x2, __fmaf_rn(w.y, x1, __fmul_rn(w.x, x0))));
}

__device__ __forceinline__ float silu(float a) { return __fmul_rn(a, sigmoidf_(a)); }

__global__ void __launch_bounds__(NT, 2) kda_scan_kernel(const __grid_constant__ ScanParams p)
{
    const int tid = threadIdx.x;
    const long long unit = blockIdx.x;              // (l * B + b) * H + h
    const int h = static_cast<int>(unit % p.H);
    const long long lb = unit / p.H;                // l * B + b
    const int b = static_cast<int>(lb % p.B);
    const int l = static_cast<int>(lb / p.B);

    int T = p.T_run;
    if (p.keep_mode == KEEP_HOST) {
        const int kp = p.keep_host[b];              // validated 1..T_rows on the host
        if (kp >= p.T_rows)
            return;                                 // full accept: resident state is final
        T = kp;
    } else if (p.keep_mode == KEEP_DEVICE) {
        const int kp = p.keep_dev[b];
        if (kp < 1 || kp > p.T_rows) {
            if (tid == 0 && h == 0 && l == 0 && p.status)
                atomicOr(p.status, KDA_ST_BADKEEP);
            return;
        }
        if (kp == p.T_rows)
            return;
        T = kp;
    }

    const int lane = tid & 31, wi = tid >> 5, hh = lane & 1, cp = lane >> 1;
    const int j0 = wi * 32 + 2 * cp;                // this thread's column pair
    const int jown = wi * 32 + lane;                // the column it finishes (j0 + hh)
    const size_t head_off = static_cast<size_t>(unit) * D * D;

    // ---- 1. state loads (in flight during the prologue) --------------------
    float2 S0[32], S1[32];  // S0[2g+r2] = (S[i][j0], S[i+1][j0]), i = 8g + 4hh + 2r2
    {
        const float *Sin = p.s_in + head_off;
#pragma unroll
        for (int g = 0; g < 16; ++g)
#pragma unroll
            for (int r2 = 0; r2 < 2; ++r2) {
                const int i = 8 * g + 4 * hh + 2 * r2;
                const float2 a = *reinterpret_cast<const float2 *>(Sin + i * D + j0);
                const float2 c = *reinterpret_cast<const float2 *>(Sin + (i + 1) * D + j0);
                S0[2 * g + r2] = make_float2(a.x, c.x);
                S1[2 * g + r2] = make_float2(a.y, c.y);
            }
    }

    // ---- 2. stage ring, raw rows and conv weights in shared memory ----------
    extern __shared__ float4 smem4[];
    const int tcap = p.keep_mode == KEEP_NONE ? p.T_run : p.T_rows;
    const int NE = T + 3;                            // ext rows per stream
    float *ext = reinterpret_cast<float *>(smem4);  // [3][NE][D]
    float4 *cw = reinterpret_cast<float4 *>(ext + 3 * (tcap + 3) * D);  // [3][D]
    float *vec = reinterpret_cast<float *>(cw + 3 * D);                  // [tcap][4][D]
    float2 *scal = reinterpret_cast<float2 *>(vec + tcap * 4 * D);       // [tcap]

    {
        const float4 *ring4 = reinterpret_cast<const float4 *>(p.ring_in + static_cast<size_t>(unit) * 9 * D);
        float4 *ext4 = reinterpret_cast<float4 *>(ext);
        for (int idx = tid; idx < 9 * D / 4; idx += NT) {
            const int s = idx / 96, rem = idx % 96, slot = rem / 32, c4 = rem % 32;
            ext4[(s * NE + slot) * 32 + c4] = ring4[idx];
        }
        const void *xs[3] = {p.xq, p.xk, p.xv};
        const size_t row0 = static_cast<size_t>(lb) * p.T_rows;  // first row of this unit
        if (p.bf16) {
            // 16 chunks of 8 bf16 per 128-channel row
            for (int idx = tid; idx < 3 * T * 16; idx += NT) {
                const int s = idx / (T * 16), rem = idx % (T * 16), t = rem / 16, q8 = rem % 16;
                const uint4 raw = *(reinterpret_cast<const uint4 *>(
                    static_cast<const uint16_t *>(xs[s]) + ((row0 + t) * p.H + h) * D) + q8);
                float4 lo, hi;
                lo.x = __uint_as_float(raw.x << 16); lo.y = __uint_as_float(raw.x & 0xffff0000u);
                lo.z = __uint_as_float(raw.y << 16); lo.w = __uint_as_float(raw.y & 0xffff0000u);
                hi.x = __uint_as_float(raw.z << 16); hi.y = __uint_as_float(raw.z & 0xffff0000u);
                hi.z = __uint_as_float(raw.w << 16); hi.w = __uint_as_float(raw.w & 0xffff0000u);
                float4 *dst = ext4 + (s * NE + 3 + t) * 32 + 2 * q8;
                dst[0] = lo;
                dst[1] = hi;
            }
        } else {
            for (int idx = tid; idx < 3 * T * 32; idx += NT) {
                const int s = idx / (T * 32), rem = idx % (T * 32), t = rem / 32, c4 = rem % 32;
                ext4[(s * NE + 3 + t) * 32 + c4] = *(reinterpret_cast<const float4 *>(
                    static_cast<const float *>(xs[s]) + ((row0 + t) * p.H + h) * D) + c4);
            }
        }
        const float4 *w4 = reinterpret_cast<const float4 *>(p.conv_w) + (static_cast<size_t>(l) * p.H + h) * 3 * D;
        for (int idx = tid; idx < 3 * D; idx += NT)
            cw[idx] = w4[idx];
    }
    __syncthreads();

    // ---- 3. prologue: one warp per row ---------------------------------------
    {
        const size_t row0 = static_cast<size_t>(lb) * p.T_rows;
        const int c0 = 4 * lane;
        for (int t = wi; t < T; t += NW) {
            float y[3][4];
#pragma unroll
            for (int s = 0; s < 3; ++s) {
                const float *e = ext + (s * NE + t) * D + c0;
                const float4 x0 = *reinterpret_cast<const float4 *>(e);
                const float4 x1 = *reinterpret_cast<const float4 *>(e + D);
                const float4 x2 = *reinterpret_cast<const float4 *>(e + 2 * D);
                const float4 x3 = *reinterpret_cast<const float4 *>(e + 3 * D);
                y[s][0] = silu(conv4(cw[s * D + c0 + 0], x0.x, x1.x, x2.x, x3.x));
                y[s][1] = silu(conv4(cw[s * D + c0 + 1], x0.y, x1.y, x2.y, x3.y));
                y[s][2] = silu(conv4(cw[s * D + c0 + 2], x0.z, x1.z, x2.z, x3.z));
                y[s][3] = silu(conv4(cw[s * D + c0 + 3], x0.w, x1.w, x2.w, x3.w));
            }
            float sq = __fmul_rn(y[0][0], y[0][0]), sk = __fmul_rn(y[1][0], y[1][0]);
#pragma unroll
            for (int cc = 1; cc < 4; ++cc) {
                sq = __fmaf_rn(y[0][cc], y[0][cc], sq);
                sk = __fmaf_rn(y[1][cc], y[1][cc], sk);
            }
            sq = warp_allsum(sq);
            sk = warp_allsum(sk);
            const float rq = rsqrtf(__fadd_rn(sq, L2_EPS));
            const float rk = rsqrtf(__fadd_rn(sk, L2_EPS));
            float qh[4], kh[4];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                qh[cc] = __fmul_rn(y[0][cc], rq);
                kh[cc] = __fmul_rn(y[1][cc], rk);
            }
            float kq = __fmul_rn(qh[0], kh[0]);
#pragma unroll
            for (int cc = 1; cc < 4; ++cc)
                kq = __fmaf_rn(qh[cc], kh[cc], kq);
            kq = warp_allsum(kq);

            const size_t rbase = ((row0 + t) * p.H + h) * D + c0;
            float dv[4];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const float rg = load_scalar(p.xg, p.bf16, rbase + cc);
                dv[cc] = expf(__fmul_rn(GATE_LOWER_BOUND, sigmoidf_(rg)));
            }
            float *vt = vec + t * 4 * D + c0;
            *reinterpret_cast<float4 *>(vt) = make_float4(dv[0], dv[1], dv[2], dv[3]);
            *reinterpret_cast<float4 *>(vt + D) = make_float4(kh[0], kh[1], kh[2], kh[3]);
            *reinterpret_cast<float4 *>(vt + 2 * D) = make_float4(qh[0], qh[1], qh[2], qh[3]);
            *reinterpret_cast<float4 *>(vt + 3 * D) = make_float4(y[2][0], y[2][1], y[2][2], y[2][3]);
            if (lane == 0) {
                const float rb = load_scalar(p.xb, p.bf16, (row0 + t) * p.H + h);
                scal[t] = make_float2(sigmoidf_(rb), kq);
            }
        }
    }
    __syncthreads();

    // ---- 4. conv ring out (+ snapshot), state snapshot -----------------------
    {
        const float4 *ext4 = reinterpret_cast<const float4 *>(ext);
        float4 *rout = reinterpret_cast<float4 *>(p.ring_out + static_cast<size_t>(unit) * 9 * D);
        float4 *rsnap = p.ring_snap ? reinterpret_cast<float4 *>(p.ring_snap + static_cast<size_t>(unit) * 9 * D) : nullptr;
        for (int idx = tid; idx < 9 * D / 4; idx += NT) {
            const int s = idx / 96, rem = idx % 96, slot = rem / 32, c4 = rem % 32;
            if (rsnap)
                rsnap[idx] = ext4[(s * NE + slot) * 32 + c4];
            rout[idx] = ext4[(s * NE + T + slot) * 32 + c4];  // last 3 of [ring, rows]
        }
    }
    if (p.s_snap) {
        float *Ss = p.s_snap + head_off;
#pragma unroll
        for (int g = 0; g < 16; ++g)
#pragma unroll
            for (int r2 = 0; r2 < 2; ++r2) {
                const int i = 8 * g + 4 * hh + 2 * r2;
                *reinterpret_cast<float2 *>(Ss + i * D + j0) = make_float2(S0[2 * g + r2].x, S1[2 * g + r2].x);
                *reinterpret_cast<float2 *>(Ss + (i + 1) * D + j0) = make_float2(S0[2 * g + r2].y, S1[2 * g + r2].y);
            }
    }

    // ---- 5. the T-row gated delta rule ---------------------------------------
    float *outp = p.out ? p.out + (static_cast<size_t>(lb) * p.T_rows * p.H + h) * D + jown : nullptr;
    for (int t = 0; t < T; ++t) {
        const float *vt = vec + t * 4 * D;
        float2 u0 = make_float2(0.f, 0.f), u1 = u0, e0 = u0, e1 = u0;
#pragma unroll
        for (int g = 0; g < 16; ++g) {
            const int ib = 8 * g + 4 * hh;
            const float4 d4 = *reinterpret_cast<const float4 *>(vt + ib);
            const float4 k4 = *reinterpret_cast<const float4 *>(vt + D + ib);
            const float4 q4 = *reinterpret_cast<const float4 *>(vt + 2 * D + ib);
            const float2 dA = make_float2(d4.x, d4.y), dB = make_float2(d4.z, d4.w);
            const float2 kA = make_float2(k4.x, k4.y), kB = make_float2(k4.z, k4.w);
            const float2 qA = make_float2(q4.x, q4.y), qB = make_float2(q4.z, q4.w);
            float2 &a0 = S0[2 * g], &a1 = S1[2 * g], &b0 = S0[2 * g + 1], &b1 = S1[2 * g + 1];
            a0 = __fmul2_rn(a0, dA);
            a1 = __fmul2_rn(a1, dA);
            b0 = __fmul2_rn(b0, dB);
            b1 = __fmul2_rn(b1, dB);
            u0 = __ffma2_rn(a0, kA, u0);
            u1 = __ffma2_rn(a1, kA, u1);
            e0 = __ffma2_rn(a0, qA, e0);
            e1 = __ffma2_rn(a1, qA, e1);
            u0 = __ffma2_rn(b0, kB, u0);
            u1 = __ffma2_rn(b1, kB, u1);
            e0 = __ffma2_rn(b0, qB, e0);
            e1 = __ffma2_rn(b1, qB, e1);
        }
        // in-thread halves, then the partner lane's 64 rows of the same column
        const float u0s = __fadd_rn(u0.x, u0.y), u1s = __fadd_rn(u1.x, u1.y);
        const float e0s = __fadd_rn(e0.x, e0.y), e1s = __fadd_rn(e1.x, e1.y);
        const float su = hh ? u0s : u1s, se = hh ? e0s : e1s;   // partner's column
        const float ku = hh ? u1s : u0s, ke = hh ? e1s : e0s;   // own column
        const float u = __fadd_rn(ku, __shfl_xor_sync(0xffffffffu, su, 1));
        const float e = __fadd_rn(ke, __shfl_xor_sync(0xffffffffu, se, 1));
        const float2 bk = scal[t];
        const float w = __fmul_rn(bk.x, __fsub_rn(vt[3 * D + jown], u));
        if (outp)
            outp[static_cast<size_t>(t) * p.H * D] = __fmul_rn(__fmaf_rn(w, bk.y, e), OUT_SCALE);
        const float wp = __shfl_xor_sync(0xffffffffu, w, 1);
        const float2 w0 = make_float2(hh ? wp : w, hh ? wp : w);
        const float2 w1 = make_float2(hh ? w : wp, hh ? w : wp);
#pragma unroll
        for (int g = 0; g < 16; ++g) {
            const float4 k4 = *reinterpret_cast<const float4 *>(vt + D + 8 * g + 4 * hh);
            const float2 kA = make_float2(k4.x, k4.y), kB = make_float2(k4.z, k4.w);
            S0[2 * g] = __ffma2_rn(kA, w0, S0[2 * g]);
            S1[2 * g] = __ffma2_rn(kA, w1, S1[2 * g]);
            S0[2 * g + 1] = __ffma2_rn(kB, w0, S0[2 * g + 1]);
            S1[2 * g + 1] = __ffma2_rn(kB, w1, S1[2 * g + 1]);
        }
    }

    // ---- 6. state write-back --------------------------------------------------
    {
        float *So = p.s_out + head_off;
#pragma unroll
        for (int g = 0; g < 16; ++g)
#pragma unroll
            for (int r2 = 0; r2 < 2; ++r2) {
                const int i = 8 * g + 4 * hh + 2 * r2;
                *reinterpret_cast<float2 *>(So + i * D + j0) = make_float2(S0[2 * g + r2].x, S1[2 * g + r2].x);
                *reinterpret_cast<float2 *>(So + (i + 1) * D + j0) = make_float2(S0[2 * g + r2].y, S1[2 * g + r2].y);
            }
    }
}

int launch_scan(const ScanParams &p, int tcap, cudaStream_t stream)
{
    const long long units = static_cast<long long>(p.L) * p.B * p.H;
    if (units == 0)
        return ok();
    if (units > 0x7fffffffLL)
        return fail(KDA_EINVAL, "L*B*H exceeds the grid limit");
    const size_t smem = smem_floats(tcap) * sizeof(float);
    static int configured_smem[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return check_launch("cudaGetDevice");
    if (dev < 64 && configured_smem[dev] < static_cast<int>(smem)) {
        const size_t need = smem_floats(KDA_TMAX) * sizeof(float);
        cudaError_t e = cudaFuncSetAttribute(kda_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(need));
        if (e != cudaSuccess)
            return fail(KDA_ECUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
        configured_smem[dev] = static_cast<int>(need);
    }
    kda_scan_kernel<<<static_cast<unsigned>(units), NT, smem, stream>>>(p);
    return check_launch("kda_scan_kernel");
}

int check_common(const kda_dims *dims, const kda_layer_state *st)
{
    if (!dims || !st)
        return fail(KDA_EINVAL, "dims and layer state must not be NULL");
    if (dims->L < 0 || dims->B < 0 || dims->H < 0)
        return fail(KDA_EINVAL, "L, B, H must be >= 0");
    if (dims->dk != D || dims->dv != D)
        return fail(KDA_EINVAL, "dk and dv must both be 128");
    if (dims->dtype != KDA_F32 && dims->dtype != KDA_BF16)
        return fail(KDA_EINVAL, "dtype must be KDA_F32 or KDA_BF16");
    if (static_cast<long long>(dims->L) * dims->B * dims->H == 0)
        return KDA_OK;  // an empty problem touches no memory; pointers may be NULL
    if (!st->state || !st->conv_ring || !st->conv_w)
        return fail(KDA_EINVAL, "state, conv_ring and conv_w must not be NULL");
    if (!aligned16(st->state) || !aligned16(st->conv_ring) || !aligned16(st->conv_w))
        return fail(KDA_EINVAL, "state, conv_ring and conv_w must be 16-byte aligned");
    return KDA_OK;
}

int check_rows(const kda_rows *rows, int dtype)
{
    if (!rows || !rows->q || !rows->k || !rows->v || !rows->g || !rows->beta)
        return fail(KDA_EINVAL, "raw rows q, k, v, g, beta must not be NULL");
    if (!aligned16(rows->q) || !aligned16(rows->k) || !aligned16(rows->v) || !aligned16(rows->g))
        return fail(KDA_EINVAL, "raw rows q, k, v, g must be 16-byte aligned");
    const uintptr_t bal = dtype == KDA_BF16 ? 1u : 3u;
    if (reinterpret_cast<uintptr_t>(rows->beta) & bal)
        return fail(KDA_EINVAL, "beta is not aligned to its element type");
    return KDA_OK;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" int kda_verify_scan(const kda_dims *dims, const kda_layer_state *st, const kda_rows *rows,
                               int T, float *out, kda_stash *stash, cudaStream_t stream)
{
    int rc = check_common(dims, st);
    if (rc)
        return rc;
    if (T < 1 || T > KDA_TMAX)
        return fail(KDA_EINVAL, "T must lie in 1..15 (K <= 14 drafts per round), got " + std::to_string(T));
    if (static_cast<long long>(dims->L) * dims->B * dims->H == 0) {
        if (stash) {
            stash->rows = rows ? *rows : kda_rows{};
            stash->T = T;
        }
        return ok();
    }
    if ((rc = check_rows(rows, dims->dtype)))
        return rc;
    if (out && (reinterpret_cast<uintptr_t>(out) & 3u))
        return fail(KDA_EINVAL, "out must be 4-byte aligned");
    if (stash) {
        if (!stash->state_snap || !stash->ring_snap)
            return fail(KDA_EINVAL, "stash->state_snap and stash->ring_snap must be allocated by the caller");
        if (!aligned16(stash->state_snap) || !aligned16(stash->ring_snap))
            return fail(KDA_EINVAL, "stash snapshots must be 16-byte aligned");
        if (stash->state_snap == st->state || stash->ring_snap == st->conv_ring)
            return fail(KDA_EINVAL, "the snapshots must not alias the resident state");
    }
    ScanParams p{};
    p.s_in = st->state;
    p.s_out = st->state;
    p.s_snap = stash ? stash->state_snap : nullptr;
    p.ring_in = st->conv_ring;
    p.ring_out = st->conv_ring;
    p.ring_snap = stash ? stash->ring_snap : nullptr;
    p.conv_w = st->conv_w;
    p.xq = rows->q; p.xk = rows->k; p.xv = rows->v; p.xg = rows->g; p.xb = rows->beta;
    p.out = out;
    p.L = dims->L; p.B = dims->B; p.H = dims->H;
    p.T_rows = T;
    p.T_run = T;
    p.bf16 = dims->dtype == KDA_BF16;
    p.keep_mode = KEEP_NONE;
    if ((rc = launch_scan(p, T, stream)))
        return rc;
    if (stash) {
        stash->rows = *rows;
        stash->T = T;
    }
    return ok();
}

extern "C" int kda_rollback(const kda_dims *dims, const kda_layer_state *st, const kda_stash *stash,
                            const int *keep, int keep_mem, int *dev_status, cudaStream_t stream)
{
    int rc = check_common(dims, st);
    if (rc)
        return rc;
    if (!stash)
        return fail(KDA_EINVAL, "stash must not be NULL");
    if (stash->T < 1 || stash->T > KDA_TMAX)
        return fail(KDA_EINVAL, "stash->T is not a verify round's row count (run kda_verify_scan first)");
    if (static_cast<long long>(dims->L) * dims->B * dims->H == 0)
        return ok();
    if (!stash->state_snap || !stash->ring_snap || !aligned16(stash->state_snap) || !aligned16(stash->ring_snap))
        return fail(KDA_EINVAL, "stash snapshots must be non-NULL and 16-byte aligned");
    if ((rc = check_rows(&stash->rows, dims->dtype)))
        return rc;
    if (!keep)
        return fail(KDA_EINVAL, "keep must not be NULL");
    ScanParams p{};
    if (keep_mem == KDA_MEM_HOST) {
        if (dims->B > KDA_HOST_KEEP_MAX)
            return fail(KDA_EINVAL, "B exceeds KDA_HOST_KEEP_MAX for a host keep array; pass keep on the device");
        bool any = false;
        for (int b = 0; b < dims->B; ++b) {
            if (keep[b] < 1 || keep[b] > stash->T)
                return fail(KDA_EINVAL, "keep[" + std::to_string(b) + "] = " + std::to_string(keep[b]) +
                                            " outside 1.." + std::to_string(stash->T) +
                                            " (the anchor row is always kept; keep = accepted drafts + 1)");
            p.keep_host[b] = static_cast<unsigned char>(keep[b]);
            any |= keep[b] < stash->T;
        }
        if (!any)
            return ok();  // every session accepted all rows: nothing to restore
        p.keep_mode = KEEP_HOST;
    } else if (keep_mem == KDA_MEM_DEVICE) {
        if (reinterpret_cast<uintptr_t>(keep) & 3u)
            return fail(KDA_EINVAL, "device keep must be 4-byte aligned");
        p.keep_mode = KEEP_DEVICE;
        p.keep_dev = keep;
    } else {
        return fail(KDA_EINVAL, "keep_mem must be KDA_MEM_HOST or KDA_MEM_DEVICE");
    }
    p.s_in = stash->state_snap;
    p.s_out = st->state;
    p.s_snap = nullptr;
    p.ring_in = stash->ring_snap;
    p.ring_out = st->conv_ring;
    p.ring_snap = nullptr;
    p.conv_w = st->conv_w;
    p.xq = stash->rows.q; p.xk = stash->rows.k; p.xv = stash->rows.v;
    p.xg = stash->rows.g; p.xb = stash->rows.beta;
    p.out = nullptr;
    p.status = dev_status;
    p.L = dims->L; p.B = dims->B; p.H = dims->H;
    p.T_rows = stash->T;
    p.T_run = stash->T;
    p.bf16 = dims->dtype == KDA_BF16;
    return launch_scan(p, stash->T, stream);
}
