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
// One CTA per session.  Every reduction and scan runs in a fixed order, so the
// results are reproducible bit for bit.  Per row: max, sum, an exact radix select
// of the k-th largest logit (four 8-bit histogram passes over order-preserving
// keys), the candidates at or above it gathered into shared memory and bitonic-
// sorted by (e descending, index ascending) for the top-p running sum, then the
// kept mass Z.  The rows stay in L1 between passes.
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
};

struct RowStats {
    float m;   // max z
    float th;  // kept iff e >= th
    float Z;   // kept mass
    int bad;   // the row holds a NaN or no finite maximum
};

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
        for (int v = threadIdx.x; v < a.V; v += SNT) {
            const unsigned key = okey(load_x(row, a.bf16, v));
            if ((key & mask) == prefix)
                atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
        }
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
    for (int v = threadIdx.x; v < a.V; v += SNT) {
        const float z = __fdiv_rn(load_x(row, a.bf16, v), a.temperature);
        nan |= z != z;
        mx = fmaxf(mx, z);
    }
    nan = block_or(sh, nan);
    const float m = block_max(sh, mx);
    if (nan || !(m > -INFINITY) || !(m < INFINITY)) {
        if (threadIdx.x == 0)
            sh.rs[slot] = RowStats{m, 0.f, 0.f, 1};
        __syncthreads();
        return;
    }
    float s = 0.f;
    for (int v = threadIdx.x; v < a.V; v += SNT)
        s = __fadd_rn(s, e_of(load_x(row, a.bf16, v), m, a.temperature));
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
            for (int v = threadIdx.x; v < a.V; v += SNT) {
                const float x = load_x(row, a.bf16, v);
                if (x >= xk) {
                    const int at = atomicAdd(&sh.ncand, 1);
                    if (at < CAP) {
                        sh.ce[at] = e_of(x, m, a.temperature);
                        sh.ci[at] = v;
                    }
                }
            }
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
    for (int v = threadIdx.x; v < a.V; v += SNT) {
        const float e = e_of(load_x(row, a.bf16, v), m, a.temperature);
        if (e >= th)
            z = __fadd_rn(z, e);
    }
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

__global__ void __launch_bounds__(SNT) sampled_accept_kernel(const SampArgs a)
{
    __shared__ Shared sh;
    const int b = blockIdx.x;
    const int K = a.T - 1;
    const size_t es = a.bf16 ? 2 : 4;
    const unsigned char *P = static_cast<const unsigned char *>(a.logits) + static_cast<size_t>(b) * a.T * a.V * es;
    const unsigned char *Q = static_cast<const unsigned char *>(a.draft_logits) + static_cast<size_t>(b) * K * a.V * es;
    int j = 0;
    bool bad = false;
    for (; j < K; ++j) {
        const int x = a.drafts[static_cast<size_t>(b) * K + j];
        row_stats(sh, a, P + static_cast<size_t>(j) * a.V * es, 0);
        row_stats(sh, a, Q + static_cast<size_t>(j) * a.V * es, 1);
        if (sh.rs[0].bad || sh.rs[1].bad) {
            bad = true;
            break;
        }
        if (threadIdx.x == 0) {
            int acc = 0;
            if (x >= 0 && x < a.V) {  // a draft id outside the vocabulary is rejected
                const float p = prob(sh.rs[0], load_x(P + static_cast<size_t>(j) * a.V * es, a.bf16, x), a.temperature);
                const float q = prob(sh.rs[1], load_x(Q + static_cast<size_t>(j) * a.V * es, a.bf16, x), a.temperature);
                const double u = a.u_accept[static_cast<size_t>(b) * K + j];
                acc = u * static_cast<double>(q) < static_cast<double>(p);
            }
            sh.flag = acc;
        }
        __syncthreads();
        if (!sh.flag)
            break;
    }
    if (!bad && j == K) {
        row_stats(sh, a, P + static_cast<size_t>(K) * a.V * es, 0);
        bad = sh.rs[0].bad;
    }
    if (bad) {
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
    const RowStats rp = sh.rs[0], rq = sh.rs[1];
    int use_resid = 0;
    if (qrow) {
        int any = 0;
        for (int v = threadIdx.x; v < a.V; v += SNT)
            any |= __fsub_rn(prob(rp, load_x(prow, a.bf16, v), a.temperature),
                             prob(rq, load_x(qrow, a.bf16, v), a.temperature)) > 0.f;
        use_resid = block_or(sh, any);
    }
    auto weight = [&](int v) -> float {
        const float p = prob(rp, load_x(prow, a.bf16, v), a.temperature);
        if (!use_resid)
            return p;
        const float r = __fsub_rn(p, prob(rq, load_x(qrow, a.bf16, v), a.temperature));
        return r > 0.f ? r : 0.f;
    };
    float w = 0.f;
    for (int v = threadIdx.x; v < a.V; v += SNT)
        w = __fadd_rn(w, weight(v));
    const float W = block_sum(sh, w);
    const float target = __fmul_rn(a.u_sample[b], W);
    // the first token whose running weight (index order, chunks of SNT) exceeds target
    float base = 0.f;
    int token = -1, last = -1;
    for (int c0 = 0; c0 < a.V && token < 0; c0 += SNT) {
        const int v = c0 + threadIdx.x;
        const float wv = v < a.V ? weight(v) : 0.f;
        float incl = wv;
        const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
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
        float wbase = 0.f;
        for (int i = 0; i < wid; ++i)
            wbase = __fadd_rn(wbase, sh.red[i]);
        float chunk = 0.f;
        for (int i = 0; i < SNW; ++i)
            chunk = __fadd_rn(chunk, sh.red[i]);
        const float run = __fadd_rn(base, __fadd_rn(wbase, incl));
        const int mine = (v < a.V && run > target) ? v : 0x7fffffff;
        const int haswt = (v < a.V && wv > 0.f) ? v : -1;
        // lowest crossing index and highest weighted index of the chunk
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

extern "C" int spec_accept_sampled(const void *logits, const void *draft_logits, int logit_dtype, int B, int T,
                                   int V, const int *drafts, const float *u_accept, const float *u_sample,
                                   const kda_sampling *sp, int *j_out, int *token_out, int *keep_out,
                                   int *dev_status, cudaStream_t stream)
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
    sampled_accept_kernel<<<B, SNT, 0, stream>>>(a);
    return check_launch("sampled_accept_kernel");
}
