// spec_sampled.cu -- sampled acceptance over the verify logits (sm_103a).
//
// glm_spec.rs (memra-engine 0.123.0), module doc SAMPLED ACCEPTANCE and
// glm5_sampled_accept / glm5_sampled_bonus: the rejection-sampling walk
//   draft r is accepted iff u_r * q~_r(x_r) < p~_r(x_r), stopping at the first
//   rejection j; then a residual draw from max(0, p~_j - q~_j) (j < K), or the
//   bonus draw from p~_K, the last verify row (j = K);
// with the target p (verify rows) and the draft q (the rows the drafts were drawn
// from) taken through the same filter (filter_stats + softmax_gather_filtered):
//   z = x / temperature, e = exp(z - max z), S = sum e; a token is kept when
//   e >= the k-th largest e (top_k), when e >= e_(n) with n the first count of
//   the descending-sorted e whose running sum reaches top_p * S (top_p), and when
//   e >= min_p (min_p); p~ = e / Z over the kept tokens.
// The uniforms are inputs; the final draw takes the first token whose running
// weight, in vocabulary order, exceeds u * (total weight).
//
// Two launches.  Every reduction and scan runs in a fixed order, so the results
// are reproducible bit for bit.
//   1. row_stats_kernel, one CTA per (session, row) of the 2T-1 target and draft
//      rows: max, sum, an exact radix select of the k-th largest logit (four 8-bit
//      histogram passes over order-preserving keys), the candidates at or above it
//      gathered into shared memory and bitonic-sorted by (e descending, index
//      ascending) for the top-p running sum, then the kept mass Z, into scratch.
//      The row stays in L1 between its passes, which read 16-byte vectors.
//   2. walk_kernel, one CTA per session: the accept tests from the row statistics,
//      then one pass for the total weight of the final draw and one scan for it.
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int SNT = 512;                   // threads per session CTA
constexpr int SNW = SNT / 32;
constexpr int CAP = 2 * KDA_SAMPLED_TOPK_MAX;  // candidates at the top-k boundary, ties included

struct SampArgs {
    const void *logits;        // [B][T][V]
    const void *draft_logits;  // [B][T-1][V]
    int bf16, B, T, V;
    const int *drafts;         // [B][T-1]
    const float *u_accept;     // [B][T-1]
    const float *u_sample;     // [B]
    float temperature, top_p, min_p;
    int top_k;
    int *j_out, *token_out, *keep_out, *status;
    int vec;  // rows start 16-byte aligned and hold a whole number of 16-byte vectors
};

struct RowStats {
    float m;   // max z
    float th;  // kept iff e >= th
    float Z;   // kept mass
    int bad;   // the row holds a NaN or no finite maximum
};
static_assert(sizeof(RowStats) == 16, "row statistics are 16 bytes in scratch");

struct Shared {
    float red[SNW];
    int ired[SNW];
    unsigned hist[256];
    float ce[CAP];
    int ci[CAP];
    int ncand;
    unsigned prefix;
    int kk;
    RowStats rs[2];
    float pick[2];
    int flag;
};

__device__ __forceinline__ float load_x(const void *row, int bf16, int v)
{
    if (bf16)
        return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const uint16_t *>(row) + v)) << 16);
    return __ldg(static_cast<const float *>(row) + v);
}

// order-preserving key of a float (larger key = larger value)
__device__ __forceinline__ unsigned okey(float x)
{
    const unsigned b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float unkey(unsigned k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// fixed-order block reductions: each thread's strided terms in order, then a tree
__device__ float block_sum(Shared &sh, float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, off));
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0)
        sh.red[w] = x;
    __syncthreads();
    float t = lane < SNW ? sh.red[lane] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, off));
    return t;
}

__device__ float block_max(Shared &sh, float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0)
        sh.red[w] = x;
    __syncthreads();
    float t = lane < SNW ? sh.red[lane] : -INFINITY;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, off));
    return t;
}

__device__ int block_or(Shared &sh, int x)
{
    return __syncthreads_or(x);
}

__device__ __forceinline__ float e_of(float x, float m, float temperature)
{
    return expf(__fsub_rn(__fdiv_rn(x, temperature), m));
}

// f(v, x) for every element of the row; each thread takes whole 16-byte vectors
// (8 bf16 or 4 f32 logits) in a fixed order where the row allows it.
template <class F>
__device__ __forceinline__ void for_row(const SampArgs &a, const void *row, F f)
{
    if (a.vec && a.bf16) {
        const uint4 *r = static_cast<const uint4 *>(row);
        for (int c = threadIdx.x; c < a.V / 8; c += SNT) {
            const uint4 u = __ldg(r + c);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                f(8 * c + 2 * m, __uint_as_float(w[m] << 16));
                f(8 * c + 2 * m + 1, __uint_as_float(w[m] & 0xffff0000u));
            }
        }
    } else if (a.vec) {
        const float4 *r = static_cast<const float4 *>(row);
        for (int c = threadIdx.x; c < a.V / 4; c += SNT) {
            const float4 u = __ldg(r + c);
            f(4 * c, u.x);
            f(4 * c + 1, u.y);
            f(4 * c + 2, u.z);
            f(4 * c + 3, u.w);
        }
    } else {
        for (int v = threadIdx.x; v < a.V; v += SNT)
            f(v, load_x(row, a.bf16, v));
    }
}

// The k-th largest logit of the row (k >= 1, k <= V), by four 8-bit radix passes.
__device__ float kth_largest(Shared &sh, const SampArgs &a, const void *row, int k)
{
    if (threadIdx.x == 0) {
        sh.prefix = 0;
        sh.kk = k;
    }
    unsigned mask = 0;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < 256; i += SNT)
            sh.hist[i] = 0;
        __syncthreads();
        const unsigned prefix = sh.prefix;
        for_row(a, row, [&](int, float x) {
            const unsigned key = okey(x);
            if ((key & mask) == prefix)
                atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
        });
        __syncthreads();
        if (threadIdx.x < 32) {  // warp 0: the bin holding the kk-th largest, from the top
            const int lane = threadIdx.x;
            unsigned c[8], tot = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = sh.hist[255 - (8 * lane + i)];
                tot += c[i];
            }
            unsigned incl = tot;  // inclusive prefix over lanes (bins counted from the top)
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off)
                    incl += y;
            }
            const unsigned excl = incl - tot;
            const int kk = sh.kk;
            const bool here = excl < static_cast<unsigned>(kk) && static_cast<unsigned>(kk) <= incl;
            if (here) {
                unsigned run = excl;
                int bin = 255 - 8 * lane;
                for (int i = 0; i < 8; ++i) {
                    if (run + c[i] >= static_cast<unsigned>(kk)) {
                        bin = 255 - (8 * lane + i);
                        break;
                    }
                    run += c[i];
                }
                sh.prefix = prefix | (static_cast<unsigned>(bin) << shift);
                sh.kk = kk - static_cast<int>(run);
            }
        }
        mask |= 255u << shift;
        __syncthreads();
    }
    return unkey(sh.prefix);
}

// Filter statistics of one row into sh.rs[slot].
__device__ void row_stats(Shared &sh, const SampArgs &a, const void *row, int slot)
{
    float mx = -INFINITY;
    int nan = 0;
    for_row(a, row, [&](int, float x) {
        const float z = __fdiv_rn(x, a.temperature);
        nan |= z != z;
        mx = fmaxf(mx, z);
    });
    nan = block_or(sh, nan);
    const float m = block_max(sh, mx);
    if (nan || !(m > -INFINITY) || !(m < INFINITY)) {
        if (threadIdx.x == 0)
            sh.rs[slot] = RowStats{m, 0.f, 0.f, 1};
        __syncthreads();
        return;
    }
    float s = 0.f;
    for_row(a, row, [&](int, float x) { s = __fadd_rn(s, e_of(x, m, a.temperature)); });
    const float S = block_sum(sh, s);
    float th = 0.f;
    if (a.top_k > 0 && a.top_k < a.V) {
        const float xk = kth_largest(sh, a, row, a.top_k);
        const float ek = e_of(xk, m, a.temperature);
        th = ek;
        if (a.top_p < 1.0f) {
            // gather every token at or above the k-th largest logit (ties included)
            if (threadIdx.x == 0)
                sh.ncand = 0;
            __syncthreads();
            for_row(a, row, [&](int v, float x) {
                if (x >= xk) {
                    const int at = atomicAdd(&sh.ncand, 1);
                    if (at < CAP) {
                        sh.ce[at] = e_of(x, m, a.temperature);
                        sh.ci[at] = v;
                    }
                }
            });
            __syncthreads();
            const int n = sh.ncand;
            if (n > CAP) {
                if (threadIdx.x == 0 && a.status)
                    atomicOr(a.status, KDA_ST_TIES);  // top-p skipped for this row
            } else {
                int np = 1;
                while (np < n)
                    np <<= 1;
                for (int i = n + threadIdx.x; i < np; i += SNT) {
                    sh.ce[i] = -1.f;
                    sh.ci[i] = 0x7fffffff;
                }
                __syncthreads();
                // bitonic sort: e descending, then index ascending
                for (int size = 2; size <= np; size <<= 1) {
                    for (int stride = size >> 1; stride > 0; stride >>= 1) {
                        for (int i = threadIdx.x; i < np; i += SNT) {
                            const int jx = i ^ stride;
                            if (jx > i) {
                                const bool up = (i & size) == 0;
                                const float e0 = sh.ce[i], e1 = sh.ce[jx];
                                const int i0 = sh.ci[i], i1 = sh.ci[jx];
                                const bool first_before = e0 > e1 || (e0 == e1 && i0 < i1);
                                if (first_before != up) {
                                    sh.ce[i] = e1;
                                    sh.ce[jx] = e0;
                                    sh.ci[i] = i1;
                                    sh.ci[jx] = i0;
                                }
                            }
                        }
                        __syncthreads();
                    }
                }
                // the running sum in sorted order (warp 0, 32 at a time, carried)
                if (threadIdx.x < 32) {
                    const float target = __fmul_rn(a.top_p, S);
                    float carry = 0.f;
                    float found = 0.f;
                    bool got = false;
                    for (int base = 0; base < n && !got; base += 32) {
                        const int i = base + static_cast<int>(threadIdx.x);
                        float incl = i < n ? sh.ce[i] : 0.f;
#pragma unroll
                        for (int off = 1; off < 32; off <<= 1) {
                            const float y = __shfl_up_sync(0xffffffffu, incl, off);
                            if (static_cast<int>(threadIdx.x) >= off)
                                incl = __fadd_rn(incl, y);
                        }
                        const float run = __fadd_rn(carry, incl);
                        const unsigned hit = __ballot_sync(0xffffffffu, i < n && run >= target);
                        if (hit) {
                            const int l = __ffs(hit) - 1;
                            found = __shfl_sync(0xffffffffu, i < n ? sh.ce[i] : 0.f, l);
                            got = true;
                        }
                        carry = __shfl_sync(0xffffffffu, run, 31);
                    }
                    if (threadIdx.x == 0)
                        sh.pick[0] = got ? found : 0.f;
                }
                __syncthreads();
                th = fmaxf(th, sh.pick[0]);
            }
        }
    }
    if (a.min_p > 0.f)
        th = fmaxf(th, a.min_p);
    float z = 0.f;
    for_row(a, row, [&](int, float x) {
        const float e = e_of(x, m, a.temperature);
        if (e >= th)
            z = __fadd_rn(z, e);
    });
    const float Z = block_sum(sh, z);
    if (threadIdx.x == 0)
        sh.rs[slot] = RowStats{m, th, Z, 0};
    __syncthreads();
}

__device__ __forceinline__ float prob(const RowStats &r, float x, float temperature)
{
    const float e = e_of(x, r.m, temperature);
    return e >= r.th ? __fdiv_rn(e, r.Z) : 0.f;
}

// Row ri of session b: target row ri (ri < T) or draft row ri - T.
__global__ void __launch_bounds__(SNT) row_stats_kernel(const SampArgs a, RowStats *__restrict__ stats)
{
    __shared__ Shared sh;
    const int nr = 2 * a.T - 1;
    const int b = blockIdx.x / nr, ri = blockIdx.x % nr;
    const int K = a.T - 1;
    const size_t es = a.bf16 ? 2 : 4;
    const unsigned char *row =
        ri < a.T ? static_cast<const unsigned char *>(a.logits) + (static_cast<size_t>(b) * a.T + ri) * a.V * es
                 : static_cast<const unsigned char *>(a.draft_logits) +
                       (static_cast<size_t>(b) * K + (ri - a.T)) * a.V * es;
    row_stats(sh, a, row, 0);
    if (threadIdx.x == 0)
        stats[blockIdx.x] = sh.rs[0];
}

__global__ void __launch_bounds__(SNT) walk_kernel(const SampArgs a, const RowStats *__restrict__ stats)
{
    __shared__ Shared sh;
    const int b = blockIdx.x;
    const int K = a.T - 1, nr = 2 * a.T - 1;
    const size_t es = a.bf16 ? 2 : 4;
    const RowStats *st = stats + static_cast<size_t>(b) * nr;
    const unsigned char *P = static_cast<const unsigned char *>(a.logits) + static_cast<size_t>(b) * a.T * a.V * es;
    const unsigned char *Q = static_cast<const unsigned char *>(a.draft_logits) + static_cast<size_t>(b) * K * a.V * es;
    if (threadIdx.x == 0) {
        int j = 0, bad = 0;
        for (; j < K; ++j) {
            const RowStats rp = st[j], rq = st[a.T + j];
            if (rp.bad || rq.bad) {
                bad = 1;
                break;
            }
            const int x = a.drafts[static_cast<size_t>(b) * K + j];
            if (x < 0 || x >= a.V)  // a draft id outside the vocabulary is rejected
                break;
            const float p = prob(rp, load_x(P + static_cast<size_t>(j) * a.V * es, a.bf16, x), a.temperature);
            const float q = prob(rq, load_x(Q + static_cast<size_t>(j) * a.V * es, a.bf16, x), a.temperature);
            const double u = a.u_accept[static_cast<size_t>(b) * K + j];
            if (!(u * static_cast<double>(q) < static_cast<double>(p)))
                break;
        }
        if (!bad && j == K && st[K].bad)
            bad = 1;
        sh.kk = j;
        sh.flag = bad;
    }
    __syncthreads();
    const int j = sh.kk;
    if (sh.flag) {
        if (threadIdx.x == 0) {
            a.j_out[b] = j;
            a.token_out[b] = -1;
            if (a.keep_out)
                a.keep_out[b] = j + 1;
            if (a.status)
                atomicOr(a.status, KDA_ST_NAN);
        }
        return;
    }
    // weights of the final draw: the residual max(0, p~_j - q~_j) (p~_j where it is
    // zero everywhere), or p~_K
    const unsigned char *prow = P + static_cast<size_t>(j) * a.V * es;
    const unsigned char *qrow = j < K ? Q + static_cast<size_t>(j) * a.V * es : nullptr;
    const RowStats rp = st[j];
    const RowStats rq = j < K ? st[a.T + j] : RowStats{0.f, 0.f, 1.f, 0};
    float wr = 0.f, wp = 0.f;
    for_row(a, prow, [&](int v, float x) {
        const float p = prob(rp, x, a.temperature);
        wp = __fadd_rn(wp, p);
        if (qrow) {
            const float r = __fsub_rn(p, prob(rq, load_x(qrow, a.bf16, v), a.temperature));
            wr = __fadd_rn(wr, r > 0.f ? r : 0.f);
        }
    });
    const float Wr = block_sum(sh, wr);
    const float Wp = block_sum(sh, wp);
    const bool use_resid = qrow && Wr > 0.f;
    const float W = use_resid ? Wr : Wp;
    const float target = __fmul_rn(a.u_sample[b], W);
    auto weight = [&](int v) -> float {
        const float p = prob(rp, load_x(prow, a.bf16, v), a.temperature);
        if (!use_resid)
            return p;
        const float r = __fsub_rn(p, prob(rq, load_x(qrow, a.bf16, v), a.temperature));
        return r > 0.f ? r : 0.f;
    };
    // the first token whose running weight (index order; chunks of SNT x 4 tokens, 4
    // consecutive tokens per thread) exceeds target
    constexpr int PER = 4;
    float base = 0.f;
    int token = -1, last = -1;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int c0 = 0; c0 < a.V && token < 0; c0 += SNT * PER) {
        const int v0 = c0 + PER * threadIdx.x;
        float wv[PER], own = 0.f;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            wv[i] = v0 + i < a.V ? weight(v0 + i) : 0.f;
            own = __fadd_rn(own, wv[i]);
        }
        float incl = own;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off)
                incl = __fadd_rn(incl, y);
        }
        __syncthreads();
        if (lane == 31)
            sh.red[wid] = incl;
        __syncthreads();
        float wbase = 0.f, chunk = 0.f;
        for (int i = 0; i < SNW; ++i) {
            if (i < wid)
                wbase = __fadd_rn(wbase, sh.red[i]);
            chunk = __fadd_rn(chunk, sh.red[i]);
        }
        const float excl_w = __shfl_up_sync(0xffffffffu, incl, 1);
        float run = __fadd_rn(base, __fadd_rn(wbase, lane ? excl_w : 0.f));
        int mine = 0x7fffffff, haswt = -1;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            run = __fadd_rn(run, wv[i]);
            if (v0 + i < a.V && run > target && mine == 0x7fffffff)
                mine = v0 + i;
            if (v0 + i < a.V && wv[i] > 0.f)
                haswt = v0 + i;
        }
        int lo = mine, hi = haswt;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
            hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
        }
        __syncthreads();
        if (lane == 0) {
            sh.ired[wid] = lo;
            sh.ci[wid] = hi;
        }
        __syncthreads();
        int clo = 0x7fffffff, chi = -1;
        for (int i = 0; i < SNW; ++i) {
            clo = min(clo, sh.ired[i]);
            chi = max(chi, sh.ci[i]);
        }
        if (clo != 0x7fffffff)
            token = clo;
        if (chi >= 0)
            last = chi;
        base = __fadd_rn(base, chunk);
    }
    if (token < 0)
        token = last;  // target rounded up to the total: the last token with weight
    if (threadIdx.x == 0) {
        a.j_out[b] = j;
        a.token_out[b] = token;
        if (a.keep_out)
            a.keep_out[b] = j + 1;
    }
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" size_t spec_accept_sampled_scratch_bytes(int B, int T)
{
    if (B <= 0 || T <= 0)
        return 0;
    return static_cast<size_t>(B) * (2 * T - 1) * sizeof(RowStats);
}

extern "C" int spec_accept_sampled(const void *logits, const void *draft_logits, int logit_dtype, int B, int T,
                                   int V, const int *drafts, const float *u_accept, const float *u_sample,
                                   const kda_sampling *sp, int *j_out, int *token_out, int *keep_out,
                                   int *dev_status, void *scratch, size_t scratch_bytes, cudaStream_t stream)
{
    if (B < 0)
        return fail(KDA_EINVAL, "B must be >= 0");
    if (T < 1 || T > KDA_TMAX)
        return fail(KDA_EINVAL, "T must lie in 1..15, got " + std::to_string(T));
    if (V < 1)
        return fail(KDA_EINVAL, "V must be >= 1");
    if (logit_dtype != KDA_F32 && logit_dtype != KDA_BF16)
        return fail(KDA_EINVAL, "logit_dtype must be KDA_F32 or KDA_BF16");
    if (!sp)
        return fail(KDA_EINVAL, "sampling parameters must not be NULL");
    if (!(sp->temperature > 0.f) || !(sp->temperature < INFINITY))
        return fail(KDA_EINVAL, "temperature must be positive and finite");
    if (sp->top_k < 0 || sp->top_k > KDA_SAMPLED_TOPK_MAX)
        return fail(KDA_EINVAL, "top_k must lie in 0..KDA_SAMPLED_TOPK_MAX");
    if (!(sp->top_p > 0.f) || sp->top_p > 1.f)
        return fail(KDA_EINVAL, "top_p must lie in (0, 1]");
    if (sp->top_p < 1.f && sp->top_k == 0)
        return fail(KDA_EINVAL, "top_p < 1 needs top_k in 1..KDA_SAMPLED_TOPK_MAX (the candidates it sorts)");
    if (!(sp->min_p >= 0.f) || !(sp->min_p < 1.f))
        return fail(KDA_EINVAL, "min_p must lie in [0, 1)");
    if (B == 0)
        return ok();
    if (!logits || !u_sample || !j_out || !token_out || (T > 1 && (!draft_logits || !drafts || !u_accept)))
        return fail(KDA_EINVAL, "logits, draft_logits, drafts, u_accept, u_sample, j_out and token_out must not "
                                "be NULL");
    const uintptr_t al = logit_dtype == KDA_BF16 ? 1u : 3u;
    if ((reinterpret_cast<uintptr_t>(logits) & al) || (reinterpret_cast<uintptr_t>(draft_logits) & al))
        return fail(KDA_EINVAL, "logits must be aligned to their element type");
    const size_t need = spec_accept_sampled_scratch_bytes(B, T);
    if (!scratch || scratch_bytes < need || !aligned16(scratch))
        return fail(KDA_EINVAL, "scratch must be 16-byte aligned device memory of at least " + std::to_string(need) +
                                    " bytes");
    if (static_cast<long long>(B) * (2 * T - 1) > 0x7fffffffLL)
        return fail(KDA_EINVAL, "B*(2T-1) exceeds the grid limit");
    SampArgs a{};
    a.logits = logits;
    a.draft_logits = draft_logits;
    a.bf16 = logit_dtype == KDA_BF16;
    a.B = B;
    a.T = T;
    a.V = V;
    a.drafts = drafts;
    a.u_accept = u_accept;
    a.u_sample = u_sample;
    a.temperature = sp->temperature;
    a.top_p = sp->top_p;
    a.min_p = sp->min_p;
    a.top_k = sp->top_k;
    a.j_out = j_out;
    a.token_out = token_out;
    a.keep_out = keep_out;
    a.status = dev_status;
    const size_t row_bytes = static_cast<size_t>(V) * (a.bf16 ? 2 : 4);
    a.vec = aligned16(logits) && (T == 1 || aligned16(draft_logits)) && row_bytes % 16 == 0;
    RowStats *stats = static_cast<RowStats *>(scratch);
    row_stats_kernel<<<static_cast<unsigned>(B * (2 * T - 1)), SNT, 0, stream>>>(a, stats);
    int rc = check_launch("row_stats_kernel");
    if (rc)
        return rc;
    walk_kernel<<<B, SNT, 0, stream>>>(a, stats);
    return check_launch("walk_kernel");
}
