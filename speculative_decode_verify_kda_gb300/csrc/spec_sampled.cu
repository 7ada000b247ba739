// spec_sampled.cu -- sampled acceptance over the verify logits (sm_103a).
//
// glm_spec.rs (memra-engine 0.123.0), module doc SAMPLED ACCEPTANCE and
// glm5_sampled_accept / glm5_sampled_bonus: the rejection-sampling walk
//   draft r is accepted iff u_r * q~_r(x_r) < p~_r(x_r), stopping at the first
//   rejection j; then a residual draw from max(0, p~_j - q~_j) (j < K), or the
//   bonus draw from p~_K, the last verify row (j = K);
// with the target p (verify rows) and the draft q (the rows the drafts were drawn
// from) taken through the same filter (filter_stats + softmax_gather_filtered):
//   z = x / temperature (f32), e = exp(z - max z) (f32), S = sum e; a token is kept
//   when e >= the k-th largest e (top_k), when e >= e_(n) with n the first count of
//   the descending-sorted e whose running sum reaches top_p * S (top_p), and when
//   e >= min_p (min_p); p~ = e / Z over the kept tokens, Z their sum.
// Precision: e is f32 (the pages' filter kernels are f32).  S, Z and every running
// sum are exact integer sums of the weights as multiples of 2^-46 (e <= 1, truncated
// to 46 fractional bits), so no sum depends on the order of its terms; the walk
// compares the f32 values of p~ and q~ in double, as the page does ((u as f64) *
// (qj as f64) < pj as f64); the final draw takes the first token, in vocabulary
// order, whose running weight exceeds u * (total weight).
// Uniforms: the caller's (spec_accept_sampled), or drawn from each session's
// Philox4x32-10 stream at its counters (spec_accept_sampled_session): accept test r
// at (uctr + r, 0, 0, 0xFFFFFFFE), the final draw at (sctr, 0, 0, 0xFFFFFFFF), under
// key (seed low, seed high); uctr advances by the tests run and sctr by one, on the
// device, so randomness never repeats across calls.
//
// Two launches.  Every reduction and scan runs in a fixed order (or on integers), so
// the results are reproducible bit for bit.
//   1. row_stats_kernel, one CTA per (session, row) of the 2T-1 target and draft
//      rows (or, when the rows' clusters fit on the GPU at once, a cluster of 8, 4 or
//      2 CTAs a row, each over a slice, merging its integer bins and sums across the
//      cluster so that every CTA takes the same decisions): max, S, an exact radix
//      select of the k-th largest logit (8-bit count passes over order-preserving
//      keys: four for f32 rows, two for bf16 rows, whose keys end in 16 fixed bits),
//      the top-p threshold by as many 8-bit passes of e-mass histograms (fixed-point
//      integer sums, per-warp bins) that find the key at which the descending running
//      sum reaches top_p * S, then the kept mass Z, into scratch.  Three sweeps of the
//      row (16-byte vectors, the row in L1 between them); the later select passes read
//      a list of the top-k candidates gathered in the second, and S is not formed when
//      bounds from the first sweep's counts prove that top-k binds (row_stats).
//   2. walk_kernel, one CTA per session (or, when the clusters fit on the GPU at once,
//      a cluster of 8, 4 or 2 CTAs a session, each weighting a slice of the draw's row):
//      the accept tests from the row statistics, then one pass for the total weight of
//      the final draw and one scan for it.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>
#include <string>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int SNT = 512;  // threads per CTA
constexpr int SNW = SNT / 32;
constexpr uint32_t TAG_ACCEPT = 0xFFFFFFFEu;    // counter word 3 of the accept-test uniforms
constexpr uint32_t TAG_DRAW = 0xFFFFFFFFu;      // counter word 3 of the residual / bonus draw

struct SampArgs {
    const void *logits;        // [B][T][V]
    const void *draft_logits;  // [B][T-1][V]
    int bf16, B, T, V;
    const int *drafts;         // [B][T-1]
    const float *u_accept;     // [B][T-1]   (caller uniforms)
    const float *u_sample;     // [B]
    const unsigned long long *seeds;  // [B]      (session streams; then u_* are unused)
    unsigned *counters;        // [B][2]: uctr, sctr, advanced in place
    float temperature, top_p, min_p;
    int top_k;
    int *j_out, *token_out, *keep_out, *status;
    int vec;  // rows start 16-byte aligned and hold a whole number of 16-byte vectors
};

struct RowStats {
    float m;     // max z
    float th;    // kept iff e >= th
    double Z;    // kept mass (its exact fixed-point sum, as a double)
    int bad;     // the row holds a NaN or no finite maximum
    float lo;    // every logit below lo has e < max(th, 2^-46): dropped, or of weight 0
    float lo_f;  // every logit below lo_f has e < th: dropped
    int pad;
};
static_assert(sizeof(RowStats) == 32, "row statistics are 32 bytes in scratch");

constexpr int SLIST = 4096;  // the candidate list of a row's top-k select, in logits

struct RowShared {
    float red[SNW];
    unsigned long long ured[SNW];
    unsigned hist[2][256];            // counts of one radix pass (alternate passes alternate)
    unsigned long long hw[SNW][256];  // per-warp e-mass bins of one radix pass
    unsigned long long tot[256];
    unsigned prefix;
    int kk, done, nlist;
    unsigned long long above;
    RowStats rs;
    // a row shared by a cluster: each CTA's part of a reduction, read by every CTA.  Each
    // scalar slot is written once; the bins alternate between two slots, so a slot is
    // written again only after a later cluster barrier, which every CTA reaches after its
    // reads of the slot: no second barrier per reduction.
    float cmax;
    int cnan;
    unsigned long long csum[4];
    unsigned long long pub[2][256];
    unsigned fine[4096];  // top-k and top-p: counts of the keys' top 12 bits (first sweep)
    int fstar;            // the fine bin holding the k-th largest
};

struct WalkShared {
    unsigned long long ured[SNW];
    int ired[SNW], ired2[SNW];
    int jsh, flag;
    float u_sample;
    float tu[KDA_TMAX], tp[KDA_TMAX], tq[KDA_TMAX];  // accept test r: its uniform, p~ and q~
    int tcode[KDA_TMAX];                             // 0 ok, 1 a NaN row, 2 draft id outside the vocabulary
    unsigned long long cw[2];                        // a cluster's session: this slice's residual and p~ weights
};

// ---- Philox4x32-10 and the session uniforms ---------------------------------------
// Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11):
// each of ten rounds multiplies counter words 0 and 2 by the round multipliers (64-bit
// products) and forms (hi(B c2) ^ c1 ^ k0, lo(B c2), hi(A c0) ^ c3 ^ k1, lo(A c0));
// the key advances by the two Weyl increments before every round but the first.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k)
{
    constexpr uint32_t A = 0xD2511F53u, B = 0xCD9E8D57u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k.x += 0x9E3779B9u;
            k.y += 0xBB67AE85u;
        }
        const uint32_t lo0 = A * c.x, hi0 = __umulhi(A, c.x);
        const uint32_t lo1 = B * c.z, hi1 = __umulhi(B, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    }
    return c;
}

// the uniform of session key `seed` at (n, 0, 0, tag): output word 0, top 24 bits x 2^-24
__device__ __forceinline__ float session_u01(unsigned long long seed, uint32_t n, uint32_t tag)
{
    const uint4 o = philox4x32_10(make_uint4(n, 0u, 0u, tag),
                                  make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)));
    return __uint2float_rn(o.x >> 8) * 5.9604644775390625e-8f;  // 2^-24, exact
}

__global__ void philox_kernel(const uint4 *__restrict__ ctr, const uint2 *__restrict__ key, uint4 *__restrict__ out,
                              int n)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        out[i] = philox4x32_10(ctr[i], key[i]);
}

// ---- row statistics -------------------------------------------------------------------
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

__device__ __forceinline__ float e_of(float x, float m, float temperature)
{
    return expf(__fsub_rn(__fdiv_rn(x, temperature), m));
}

// a weight in [0, 1] as an integer multiple of 2^-46 (truncated): exact integer sums,
// so no sum depends on the order of its additions.  Formed from the float's fields
// with integer shifts (a float-to-64-bit conversion runs on the FP64 pipe, which is
// narrow on this GPU): e = m 2^(E - 150) with m the 24-bit significand, so
// e 2^46 = m 2^(E - 104).
__device__ __forceinline__ unsigned long long fx(float e)
{
    const uint32_t b = __float_as_uint(e);
    const int E = static_cast<int>(b >> 23);
    if (E < 81)  // below 2^-46, or zero
        return 0ull;
    const unsigned long long m = (b & 0x7fffffu) | 0x800000u;
    return E >= 104 ? m << (E - 104) : m >> (104 - E);
}
constexpr double FX_UNIT = 1.4210854715202004e-14;  // 2^-46

// block reductions: integer sums (any order gives the same result) and the maximum
__device__ unsigned long long block_sum_u64(unsigned long long *red, unsigned long long x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, off);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0)
        red[w] = x;
    __syncthreads();
    unsigned long long t = lane < SNW ? red[lane] : 0ull;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        t += __shfl_xor_sync(0xffffffffu, t, off);
    return t;
}

__device__ float block_max(float *red, float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0)
        red[w] = x;
    __syncthreads();
    float t = lane < SNW ? red[lane] : -INFINITY;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, off));
    return t;
}

__device__ __forceinline__ int row_chunks(const SampArgs &a);

// The chunks of a row that CTA `rank` of a cluster of CL takes (all of them when CL = 1).
template <int CL>
__device__ __forceinline__ void slice_of(const SampArgs &a, int &c0, int &c1)
{
    const int nc = row_chunks(a);
    if (CL == 1) {
        c0 = 0;
        c1 = nc;
        return;
    }
    const int rank = static_cast<int>(cooperative_groups::this_cluster().block_rank());
    c0 = static_cast<int>(static_cast<long long>(nc) * rank / CL);
    c1 = static_cast<int>(static_cast<long long>(nc) * (rank + 1) / CL);
}

// f(v, x) for every element of the CTA's slice of the row; each thread takes whole
// 16-byte vectors (8 bf16 or 4 f32 logits) in a fixed order where the row allows it.
template <int CL, class F>
__device__ __forceinline__ void for_row(const SampArgs &a, const void *row, F f)
{
    int c0, c1;
    slice_of<CL>(a, c0, c1);
    if (a.vec && a.bf16) {
        const uint4 *r = static_cast<const uint4 *>(row);
        for (int c = c0 + threadIdx.x; c < c1; c += SNT) {
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
        for (int c = c0 + threadIdx.x; c < c1; c += SNT) {
            const float4 u = __ldg(r + c);
            f(4 * c, u.x);
            f(4 * c + 1, u.y);
            f(4 * c + 2, u.z);
            f(4 * c + 3, u.w);
        }
    } else {
        for (int v = c0 + threadIdx.x; v < c1; v += SNT)
            f(v, load_x(row, a.bf16, v));
    }
}

// ---- reductions over the CTAs of a cluster that share a row ------------------------
// Each CTA publishes its part in its own shared memory; after a cluster barrier every CTA
// reads all parts in rank order, so every CTA holds the same (exact or order-fixed)
// result.  A published slot is not written again before a later barrier (see RowShared),
// and the kernel ends with a barrier, so no CTA leaves while another reads its parts.

// the NaN flag and the maximum of the row, in one exchange
template <int CL>
__device__ void cluster_or_max(RowShared &sh, int &nan, float &m)
{
    if (CL == 1)
        return;
    auto cl = cooperative_groups::this_cluster();
    if (threadIdx.x == 0) {
        sh.cnan = nan;
        sh.cmax = m;
    }
    cl.sync();
    int o = 0;
    float x = -INFINITY;
    for (int r = 0; r < CL; ++r) {
        o |= *cl.map_shared_rank(&sh.cnan, r);
        x = fmaxf(x, *cl.map_shared_rank(&sh.cmax, r));
    }
    nan = o;
    m = x;
}

// slot: 0 to 3, each used once per row
template <int CL>
__device__ unsigned long long cluster_sum(RowShared &sh, unsigned long long x, int slot)
{
    if (CL == 1)
        return x;
    auto cl = cooperative_groups::this_cluster();
    if (threadIdx.x == 0)
        sh.csum[slot] = x;
    cl.sync();
    unsigned long long t = 0;
    for (int r = 0; r < CL; ++r)
        t += *cl.map_shared_rank(&sh.csum[slot], r);
    return t;
}

// bins[0..256) of every CTA of the cluster summed into out[0..256) of each (integer
// sums); the caller's bins are complete, and stay unwritten until the next barrier
template <int CL, class U>
__device__ void cluster_bins(const U *bins, U *out)
{
    if (CL == 1)
        return;
    auto cl = cooperative_groups::this_cluster();
    cl.sync();
    for (int i = threadIdx.x; i < 256; i += SNT) {
        U t = 0;
        for (int r = 0; r < CL; ++r)
            t += cl.map_shared_rank(bins, r)[i];
        out[i] = t;
    }
}

// The low 16 bits of the keys of bf16 logits: zero for a positive value, all ones for a
// negative one (the key complements a negative float).  Keys that share their top 16 bits
// are then the same key, so the two low radix passes of a bf16 row are skipped.
__device__ __forceinline__ unsigned bf16_key_low(unsigned prefix)
{
    return (prefix & 0x80000000u) ? 0u : 0xffffu;
}

// The same traversal as for_row, chunk by chunk: chunk c of the row into xs[0..n), the
// elements for_row hands thread threadIdx.x in that order.
__device__ __forceinline__ int row_chunks(const SampArgs &a)
{
    return a.vec ? (a.bf16 ? a.V / 8 : a.V / 4) : a.V;
}

__device__ __forceinline__ int load_chunk(const SampArgs &a, const void *row, int c, float (&xs)[8])
{
    if (a.vec && a.bf16) {
        const uint4 u = __ldg(static_cast<const uint4 *>(row) + c);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            xs[2 * m] = __uint_as_float(w[m] << 16);
            xs[2 * m + 1] = __uint_as_float(w[m] & 0xffff0000u);
        }
        return 8;
    }
    if (a.vec) {
        const float4 u = __ldg(static_cast<const float4 *>(row) + c);
        xs[0] = u.x;
        xs[1] = u.y;
        xs[2] = u.z;
        xs[3] = u.w;
        return 4;
    }
    xs[0] = load_x(row, a.bf16, c);
    return 1;
}

// Runs of one bin counted in a register and added to the bins once per run (a thread's
// consecutive logits mostly share the top bytes of their keys).
struct BinRun {
    int cur = -1;
    unsigned run = 0;
    __device__ __forceinline__ void add(unsigned *hist, int bin)
    {
        if (bin != cur) {
            if (cur >= 0)
                atomicAdd(&hist[cur], run);
            cur = bin;
            run = 0;
        }
        ++run;
    }
    __device__ __forceinline__ void flush(unsigned *hist)
    {
        if (cur >= 0)
            atomicAdd(&hist[cur], run);
    }
};

// The CTA's logits handed to f(x): the candidate list when it holds them (n >= 0), else
// the CTA's slice of the row.
template <int CL, class F>
__device__ __forceinline__ void each_logit(const SampArgs &a, const void *row, const float *list, int n, F f)
{
    if (n >= 0) {
        for (int i = threadIdx.x; i < n; i += SNT)
            f(list[i]);
    } else {
        for_row<CL>(a, row, [&](int, float x) { f(x); });
    }
}

// One step of the exact select of the k-th largest key: hist holds this CTA's counts of
// the byte at `shift` of the keys under `prefix` (complete: a barrier of the CTA precedes
// the call); warp 0 finds the bin holding the sh.kk-th largest, counting from the top,
// and extends sh.prefix by it.
template <int CL>
__device__ void pick_kth_bin(RowShared &sh, const unsigned *hist, unsigned prefix, int shift)
{
    const unsigned *cnt = hist;
    if (CL > 1) {  // a cluster's row: the counts of every slice (into the spare e-mass bins)
        cluster_bins<CL>(hist, reinterpret_cast<unsigned *>(&sh.tot[0]));
        __syncthreads();
        cnt = reinterpret_cast<const unsigned *>(&sh.tot[0]);
    }
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        unsigned c[8], tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c[i] = cnt[255 - (8 * lane + i)];
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
        if (excl < static_cast<unsigned>(kk) && static_cast<unsigned>(kk) <= incl) {
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
    __syncthreads();
}

// The key of the top-p boundary: the largest key kappa whose mass F(kappa) = sum of e
// over the tokens with key >= kappa reaches `target` (top_p * S, in fixed-point units).
// Tokens in key order are tokens in e order, so kappa is the key of the token at which
// the descending running sum first reaches the target, and e(kappa) is the threshold.
// Four 8-bit passes from the top byte; each pass bins the e-mass of the tokens under the
// current prefix, and warp 0 walks the bins from the top (above: the mass of the keys
// already passed).  Only keys >= floor take part (the k-th largest key under top_k):
// when their whole mass stays below the target, the top-p threshold lies under the
// top-k one and floor is returned.  The passes read the candidate list when it holds
// every key >= floor (nl >= 0), else the row.
template <int CL>
__device__ unsigned topp_key(RowShared &sh, const SampArgs &a, const void *row, const float *list, int nl, float m,
                             double target, unsigned floor)
{
    const int w = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        sh.prefix = 0;
        sh.above = 0;
        sh.done = 0;
    }
    unsigned mask = 0;
    const int passes = a.bf16 ? 2 : 4;
    for (int pass = 0; pass < passes; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < SNW * 256; i += SNT)
            (&sh.hw[0][0])[i] = 0;
        __syncthreads();
        const unsigned prefix = sh.prefix;
        // runs of one bin summed in a register (integer sums: the order does not matter)
        int cur = -1;
        unsigned long long run = 0;
        each_logit<CL>(a, row, list, nl, [&](float x) {
            const unsigned key = okey(x);
            if ((key & mask) != prefix || key < floor)
                return;
            const int bin = static_cast<int>((key >> shift) & 255u);
            if (bin != cur) {
                if (cur >= 0)
                    atomicAdd(&sh.hw[w][cur], run);
                cur = bin;
                run = 0;
            }
            run += fx(e_of(x, m, a.temperature));
        });
        if (cur >= 0)
            atomicAdd(&sh.hw[w][cur], run);
        __syncthreads();
        // the CTA's bins (a cluster's row: published, then the bins of every slice summed)
        unsigned long long *mine = CL > 1 ? sh.pub[pass & 1] : sh.tot;
        for (int d = threadIdx.x; d < 256; d += SNT) {
            unsigned long long t = 0;
            for (int i = 0; i < SNW; ++i)
                t += sh.hw[i][d];
            mine[d] = t;
        }
        __syncthreads();
        if (CL > 1) {
            cluster_bins<CL>(static_cast<const unsigned long long *>(mine), sh.tot);
            __syncthreads();
        }
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            const unsigned long long above = sh.above;
            unsigned long long c[8], tot = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = sh.tot[255 - (8 * lane + i)];
                tot += c[i];
            }
            unsigned long long incl = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off)
                    incl += y;
            }
            const unsigned long long excl = incl - tot;
            const unsigned long long all = __shfl_sync(0xffffffffu, incl, 31);
            if (pass == 0 && static_cast<double>(all) < target) {  // top-k binds
                if (lane == 0) {
                    sh.prefix = floor;
                    sh.done = 1;
                }
                __syncwarp();
            }
            const bool here = !sh.done && static_cast<double>(above + excl) < target &&
                              static_cast<double>(above + incl) >= target;
            const unsigned hit = __ballot_sync(0xffffffffu, here);
            if (here) {
                unsigned long long run = excl;
                int bin = 255 - (8 * lane + 7);
                for (int i = 0; i < 8; ++i) {
                    if (static_cast<double>(above + run + c[i]) >= target) {
                        bin = 255 - (8 * lane + i);
                        break;
                    }
                    run += c[i];
                }
                sh.prefix = prefix | (static_cast<unsigned>(bin) << shift);
                sh.above = above + run;
            }
            if (!hit && !sh.done && lane == 0) {  // rounding left the target above the mass: the lowest bin with mass
                int bin = 0;
                while (bin < 255 && sh.tot[bin] == 0)
                    ++bin;
                unsigned long long run = 0;
                for (int d = 255; d > bin; --d)
                    run += sh.tot[d];
                sh.prefix = prefix | (static_cast<unsigned>(bin) << shift);
                sh.above = above + run;
            }
        }
        mask |= 255u << shift;
        __syncthreads();
        if (sh.done)
            return sh.prefix;
    }
    // (a chosen group always holds mass, so a bf16 row's low passes would pick its one key)
    return a.bf16 ? sh.prefix | bf16_key_low(sh.prefix) : sh.prefix;
}

// A logit below which every e lies under te (> 0): x -> RN(RN(x / t) - m) is
// non-decreasing, exp is increasing and expf lies within 2 ulp (2^-22 relative) of exp,
// so a logit c whose e lies below te (1 - 2^-20) bounds the e of every smaller logit
// below te.  The candidates start near the logit whose e is te and step down; -inf when
// none checks out (or te <= 0).  Every thread computes the same value.
__device__ float skip_below(float m, float te, float temperature)
{
    if (!(te > 0.f))
        return -INFINITY;
    const float bound = te * (1.f - 0x1p-20f);
    float c = __fmul_rn(temperature, __fadd_rn(m, logf(te)));
    float step = fmaxf(fabsf(c), 1.f) * 0x1p-10f;
    for (int i = 0; i < 6; ++i, step *= 8.f) {
        if (!(c > -INFINITY) || !(c < INFINITY))
            break;
        if (e_of(c, m, temperature) < bound)
            return c;
        c = __fsub_rn(c, step);
    }
    return -INFINITY;
}

// Filter statistics of one row into sh.rs (CL > 1: the row shared by the CTAs of a
// cluster, each taking a slice; every CTA ends with the same statistics).  Sweeps of the
// CTA's logits: (1) the maximum, the NaN flag and the first count pass of the top-k
// select; (2) with top-k, the candidates: every logit whose key's top byte is at or above
// the one holding the k-th largest (every later pass selects among them), into `list`
// when their count, known from the first pass, fits (else the later passes read the row
// again), and S for top-p; (3) the kept mass Z.  All sums and counts are integers, so the
// order in which the list holds the candidates does not matter.
// Top-k and top-p together: the first pass counts the keys' top 12 bits (bins of an
// eighth of a binade); from those counts, S is bounded from below (every logit of a bin
// is at least the bin's smallest value) and the mass of the top-k set from above (every
// key >= the k-th largest lies in its bin or a higher one, every logit of a bin is at
// most the bin's largest value), the e of a bin's edge taken with a 2^-19 margin for
// expf's 2-ulp error.  When the bound of the top-k mass stays below top_p times the
// bound of S, top-k binds: top-p's threshold lies under the top-k one, and S is not formed.
template <int CL>
__device__ void row_stats(RowShared &sh, float *list, const SampArgs &a, const void *row)
{
    const bool topk = a.top_k > 0 && a.top_k < a.V, topp = a.top_p < 1.0f;
    const bool fine = topk && topp;
    const int passes = a.bf16 ? 2 : 4;
    if (fine)
        for (int i = threadIdx.x; i < 4096; i += SNT)
            sh.fine[i] = 0;
    else if (topk)
        for (int i = threadIdx.x; i < 256; i += SNT)
            sh.hist[0][i] = 0;
    if (threadIdx.x == 0) {
        sh.prefix = 0;
        sh.kk = a.top_k;
        sh.nlist = 0;
    }
    __syncthreads();
    float mx = -INFINITY;
    int nan = 0;
    BinRun br;
    unsigned *const h0 = fine ? sh.fine : sh.hist[0];
    const int hs = fine ? 20 : 24;
    for_row<CL>(a, row, [&](int, float x) {
        nan |= x != x;
        mx = fmaxf(mx, x);
        if (topk)
            br.add(h0, static_cast<int>(okey(x) >> hs));
    });
    br.flush(h0);
    nan = __syncthreads_or(nan);
    float m = block_max(sh.red, mx);
    cluster_or_max<CL>(sh, nan, m);
    // x -> RN(x / t) is non-decreasing for t > 0, so the largest z is z of the largest
    // logit (and z is NaN exactly where x is)
    m = __fdiv_rn(m, a.temperature);
    if (nan || !(m > -INFINITY) || !(m < INFINITY)) {
        if (threadIdx.x == 0)
            sh.rs = RowStats{m, 0.f, 0.0, 1, -INFINITY, -INFINITY, 0};
        __syncthreads();
        return;
    }
    bool gather = false, skip_s = false;
    if (topk) {
        if (fine) {  // the top bytes' counts from the fine ones
            for (int b = threadIdx.x; b < 256; b += SNT) {
                unsigned c = 0;
                for (int i = 0; i < 16; ++i)
                    c += sh.fine[16 * b + i];
                sh.hist[0][b] = c;
            }
            __syncthreads();
        }
        pick_kth_bin<CL>(sh, sh.hist[0], 0u, 24);
        const unsigned bin0 = sh.prefix >> 24;
        unsigned long long n_part = 0;  // this CTA's candidates
        for (int b = threadIdx.x; b < 256; b += SNT)
            if (static_cast<unsigned>(b) >= bin0)
                n_part += sh.hist[0][b];
        gather = block_sum_u64(sh.ured, n_part) <= static_cast<unsigned long long>(SLIST);
        if (fine) {
            if (threadIdx.x < 32) {  // the fine bin of bin0 holding the kk-th largest (the row's counts)
                const int lane = threadIdx.x;
                unsigned c = 0;
                if (lane < 16) {
                    const int f = 16 * static_cast<int>(bin0) + 15 - lane;  // from the top
                    if (CL > 1) {
                        auto cl = cooperative_groups::this_cluster();
                        for (int r = 0; r < CL; ++r)
                            c += cl.map_shared_rank(sh.fine, r)[f];
                    } else {
                        c = sh.fine[f];
                    }
                }
                unsigned incl = c;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const unsigned y = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off)
                        incl += y;
                }
                const unsigned kk = static_cast<unsigned>(sh.kk);
                if (lane < 16 && incl - c < kk && kk <= incl)
                    sh.fstar = 16 * static_cast<int>(bin0) + 15 - lane;
            }
            __syncthreads();
            const int fs = sh.fstar;
            unsigned long long lo_part = 0, hi_part = 0;
            for (int f = threadIdx.x; f < 4096; f += SNT) {
                const unsigned c = sh.fine[f];
                if (!c)
                    continue;
                const unsigned fu = static_cast<unsigned>(f);
                const float x0 = unkey(fu << 20), x1 = unkey(((fu + 1u) << 20) - 1u);  // the bin's edges
                if (x0 > -INFINITY && x0 < INFINITY)
                    lo_part += static_cast<unsigned long long>(c) *
                               fx(__fmul_rn(e_of(x0, m, a.temperature), 1.f - 0x1p-19f));
                if (f >= fs) {
                    float e1 = 1.f;
                    if (x1 > -INFINITY && x1 < INFINITY)
                        e1 = fminf(e_of(x1, m, a.temperature), 1.f);
                    hi_part += static_cast<unsigned long long>(c) * fx(__fmul_rn(e1, 1.f + 0x1p-19f));
                }
            }
            const unsigned long long s_lo = cluster_sum<CL>(sh, block_sum_u64(sh.ured, lo_part), 2);
            const unsigned long long mk_hi = cluster_sum<CL>(sh, block_sum_u64(sh.ured, hi_part), 3);
            skip_s = static_cast<double>(mk_hi) < static_cast<double>(a.top_p) * static_cast<double>(s_lo);
        }
    }
    const unsigned base = sh.prefix;
    const bool need_s = topp && !skip_s;
    unsigned long long s = 0;
    if (gather || need_s)
        for_row<CL>(a, row, [&](int, float x) {
            if (need_s)
                s += fx(e_of(x, m, a.temperature));
            if (gather && okey(x) >= base)
                list[atomicAdd(&sh.nlist, 1)] = x;  // (the count fits: see above)
        });
    __syncthreads();
    const int nl = gather ? sh.nlist : -1;
    float th = 0.f;
    unsigned floor = 0;  // the k-th largest key: top-p looks no lower
    if (topk) {
        unsigned mask = 0xff000000u;
        for (int pass = 1; pass < passes; ++pass) {  // (bf16 keys end in 16 fixed bits)
            const int shift = 24 - 8 * pass;
            unsigned *hist = sh.hist[pass & 1];
            for (int i = threadIdx.x; i < 256; i += SNT)
                hist[i] = 0;
            __syncthreads();
            const unsigned prefix = sh.prefix;
            BinRun r;
            each_logit<CL>(a, row, list, nl, [&](float x) {
                const unsigned key = okey(x);
                if ((key & mask) == prefix)
                    r.add(hist, static_cast<int>((key >> shift) & 255u));
            });
            r.flush(hist);
            __syncthreads();
            pick_kth_bin<CL>(sh, hist, prefix, shift);
            mask |= 255u << shift;
        }
        floor = a.bf16 ? sh.prefix | bf16_key_low(sh.prefix) : sh.prefix;
        th = e_of(unkey(floor), m, a.temperature);
    }
    if (need_s) {
        const unsigned long long S = cluster_sum<CL>(sh, block_sum_u64(sh.ured, s), 0);
        const double target = static_cast<double>(a.top_p) * static_cast<double>(S);
        th = fmaxf(th, e_of(unkey(topp_key<CL>(sh, a, row, list, nl, m, target, floor)), m, a.temperature));
    }
    if (a.min_p > 0.f)
        th = fmaxf(th, a.min_p);
    const float lo = skip_below(m, fmaxf(th, 0x1p-46f), a.temperature);
    unsigned long long z = 0;
    for_row<CL>(a, row, [&](int, float x) {
        if (x >= lo) {  // (a logit below lo is dropped or weighs 0)
            const float e = e_of(x, m, a.temperature);
            if (e >= th)
                z += fx(e);
        }
    });
    const double Z = static_cast<double>(cluster_sum<CL>(sh, block_sum_u64(sh.ured, z), 1)) * FX_UNIT;
    if (threadIdx.x == 0)
        sh.rs = RowStats{m, th, Z, 0, lo, skip_below(m, th, a.temperature), 0};
    __syncthreads();
}

// p~ of logit x under row statistics r, as the f32 value the walk compares
__device__ __forceinline__ float prob32(const RowStats &r, float x, float temperature)
{
    const float e = e_of(x, r.m, temperature);
    return e >= r.th ? __double2float_rn(__ddiv_rn(static_cast<double>(e), r.Z)) : 0.f;
}

// Row ri of session b: target row ri (ri < T) or draft row ri - T.
__device__ __forceinline__ const void *stats_row(const SampArgs &a, int rowi)
{
    const int nr = 2 * a.T - 1;
    const int b = rowi / nr, ri = rowi % nr;
    const int K = a.T - 1;
    const size_t es = a.bf16 ? 2 : 4;
    return ri < a.T ? static_cast<const unsigned char *>(a.logits) + (static_cast<size_t>(b) * a.T + ri) * a.V * es
                    : static_cast<const unsigned char *>(a.draft_logits) +
                          (static_cast<size_t>(b) * K + (ri - a.T)) * a.V * es;
}

// The launches' dynamic shared memory: the row's work space, then the candidate list.
constexpr size_t ROW_SMEM = sizeof(RowShared) + SLIST * sizeof(float);

// One CTA a row (many rows: the GPU is full).
__global__ void __launch_bounds__(SNT) row_stats_kernel(const SampArgs a, RowStats *__restrict__ stats)
{
    extern __shared__ __align__(16) unsigned char smem[];
    RowShared &sh = *reinterpret_cast<RowShared *>(smem);
    row_stats<1>(sh, reinterpret_cast<float *>(smem + sizeof(RowShared)), a, stats_row(a, blockIdx.x));
    if (threadIdx.x == 0)
        stats[blockIdx.x] = sh.rs;
}

// A cluster of CL CTAs a row, each over a slice of it (few rows: one CTA a row would
// leave most SMs idle and run every pass of the row on one).
template <int CL>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(SNT, 1)
    row_stats_cluster_kernel(const SampArgs a, RowStats *__restrict__ stats)
{
    extern __shared__ __align__(16) unsigned char smem[];
    RowShared &sh = *reinterpret_cast<RowShared *>(smem);
    const int rowi = blockIdx.x / CL;
    row_stats<CL>(sh, reinterpret_cast<float *>(smem + sizeof(RowShared)), a, stats_row(a, rowi));
    auto cl = cooperative_groups::this_cluster();
    if (threadIdx.x == 0 && cl.block_rank() == 0)
        stats[rowi] = sh.rs;
    cl.sync();  // the CTA's published parts stay until every CTA has read them
}

// the two halves of a cluster barrier: arrive (release) and wait (acquire)
__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The walk of session b.  CL > 1: the draw's row shared by a cluster of CL CTAs, each
// weighting a slice of it.  Every CTA runs the accept tests (the same inputs give the
// same j), the slices' weight sums are exchanged, and the CTA whose slice holds the
// draw's target (or, for a target rounded up to the total, the last slice with weight)
// walks its slice and writes the results.
template <int CL>
__device__ void walk_session(WalkShared &sh, const SampArgs &a, const RowStats *__restrict__ stats, int b)
{
    const int K = a.T - 1, nr = 2 * a.T - 1;
    const size_t es = a.bf16 ? 2 : 4;
    const RowStats *st = stats + static_cast<size_t>(b) * nr;
    const unsigned char *P = static_cast<const unsigned char *>(a.logits) + static_cast<size_t>(b) * a.T * a.V * es;
    const unsigned char *Q = static_cast<const unsigned char *>(a.draft_logits) + static_cast<size_t>(b) * K * a.V * es;
    const bool session = a.seeds != nullptr;
    const unsigned long long seed = session ? a.seeds[b] : 0ull;
    const uint32_t uctr = session ? a.counters[2 * b] : 0u, sctr = session ? a.counters[2 * b + 1] : 0u;
    const int rank = CL > 1 ? static_cast<int>(cooperative_groups::this_cluster().block_rank()) : 0;
    // every accept test's inputs at once (thread r: test r), then the walk in order
    if (threadIdx.x < K) {
        const int r = threadIdx.x;
        const RowStats rp = st[r], rq = st[a.T + r];
        const int x = a.drafts[static_cast<size_t>(b) * K + r];
        sh.tu[r] = session ? session_u01(seed, uctr + static_cast<uint32_t>(r), TAG_ACCEPT)
                           : a.u_accept[static_cast<size_t>(b) * K + r];
        sh.tcode[r] = rp.bad || rq.bad ? 1 : (x < 0 || x >= a.V ? 2 : 0);
        if (sh.tcode[r] == 0) {
            sh.tp[r] = prob32(rp, load_x(P + static_cast<size_t>(r) * a.V * es, a.bf16, x), a.temperature);
            sh.tq[r] = prob32(rq, load_x(Q + static_cast<size_t>(r) * a.V * es, a.bf16, x), a.temperature);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int j = 0, bad = 0;
        for (; j < K; ++j) {
            if (sh.tcode[j] == 1) {
                bad = 1;
                break;
            }
            if (sh.tcode[j] == 2)  // a draft id outside the vocabulary is rejected
                break;
            if (!(static_cast<double>(sh.tu[j]) * static_cast<double>(sh.tq[j]) < static_cast<double>(sh.tp[j])))
                break;
        }
        if (!bad && j == K && st[K].bad)
            bad = 1;
        sh.jsh = j;
        sh.flag = bad;
        sh.u_sample = session ? session_u01(seed, sctr, TAG_DRAW) : a.u_sample[b];
    }
    __syncthreads();
    const int j = sh.jsh;
    // the results, by thread 0 of the one CTA that writes them; the counters advance by
    // the tests run (j + 1 on a rejection, K when every draft passed) and one draw (a
    // cluster's CTAs have all read them: a cluster barrier precedes every write)
    auto finish = [&](int token) {
        a.j_out[b] = j;
        a.token_out[b] = token;
        if (a.keep_out)
            a.keep_out[b] = j + 1;
        if (session) {
            a.counters[2 * b] = uctr + static_cast<uint32_t>(j < K ? j + 1 : K);
            a.counters[2 * b + 1] = sctr + 1u;
        }
    };
    if (sh.flag) {
        if (CL > 1)
            cooperative_groups::this_cluster().sync();
        if (threadIdx.x == 0 && rank == 0) {
            finish(-1);
            if (a.status)
                atomicOr(a.status, KDA_ST_NAN);
        }
        return;
    }
    // weights of the final draw as fixed-point integers: the residual max(0, p~_j - q~_j)
    // (p~_j where it is zero everywhere), or p~_K scaled by its mass (e itself)
    const unsigned char *prow = P + static_cast<size_t>(j) * a.V * es;
    const unsigned char *qrow = j < K ? Q + static_cast<size_t>(j) * a.V * es : nullptr;
    const RowStats rp = st[j];
    const RowStats rq = j < K ? st[a.T + j] : RowStats{0.f, 0.f, 1.0, 0, -INFINITY, -INFINITY, 0};
    const float ip = __double2float_rn(1.0 / rp.Z), iq = __double2float_rn(1.0 / rq.Z);
    // (below rp.lo a target logit is dropped or its p~ and residual weigh 0, p~ <= e
    // as Z >= 1; below rq.lo_f a draft logit is dropped: the weights are those of the
    // full evaluation)
    auto wp_of = [&](float x) -> unsigned long long {
        if (!(x >= rp.lo))
            return 0ull;
        const float e = e_of(x, rp.m, a.temperature);
        return e >= rp.th ? fx(e) : 0ull;
    };
    auto wr_of = [&](float x, float xq) -> unsigned long long {
        float pt = 0.f, qt = 0.f;
        if (x >= rp.lo) {
            const float ep = e_of(x, rp.m, a.temperature);
            if (ep >= rp.th)
                pt = __fmul_rn(ep, ip);
        }
        if (xq >= rq.lo_f) {
            const float eq = e_of(xq, rq.m, a.temperature);
            if (eq >= rq.th)
                qt = __fmul_rn(eq, iq);
        }
        const float r = __fsub_rn(pt, qt);
        return r > 0.f ? fx(r) : 0ull;
    };
    // thread t owns a contiguous run of the slice's 16-byte chunks (the for_row chunks):
    // one pass sums both weight kinds per run; the block's exclusive scan of the run sums
    // finds the run holding the target, and its thread walks it
    const int per = a.vec ? (a.bf16 ? 8 : 4) : 1;
    int s0, s1;
    slice_of<CL>(a, s0, s1);
    const int cs = (s1 - s0 + SNT - 1) / SNT;
    const int c0 = s0 + threadIdx.x * cs, c1 = min(s1, c0 + cs);
    unsigned long long sr = 0, sp = 0;
    for (int c = c0; c < c1; ++c) {
        float xp[8], xq[8];
        const int n = load_chunk(a, prow, c, xp);
        if (qrow)
            load_chunk(a, qrow, c, xq);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < n) {
                sp += wp_of(xp[i]);
                if (qrow)
                    sr += wr_of(xp[i], xq[i]);
            }
    }
    unsigned long long Wr = block_sum_u64(sh.ured, sr);
    unsigned long long Wp = block_sum_u64(sh.ured, sp);
    // the slice's weights, the weight of the slices before it, the last slice with weight
    unsigned long long cr = Wr, cp = Wp, br = 0, bp = 0;
    int lr = 0, lp = 0;
    if (CL > 1) {
        auto cl = cooperative_groups::this_cluster();
        if (threadIdx.x == 0) {
            sh.cw[0] = Wr;
            sh.cw[1] = Wp;
        }
        cl.sync();
        Wr = Wp = 0;
        lr = lp = -1;
        for (int r = 0; r < CL; ++r) {
            const unsigned long long *o = cl.map_shared_rank(sh.cw, r);
            const unsigned long long xr = o[0], xq = o[1];
            if (r < rank) {
                br += xr;
                bp += xq;
            }
            if (xr)
                lr = r;
            if (xq)
                lp = r;
            Wr += xr;
            Wp += xq;
        }
        cluster_arrive();  // this CTA has read the parts (the matching wait ends the kernel)
    }
    const bool use_resid = qrow && Wr > 0;
    const unsigned long long W = use_resid ? Wr : Wp, own = use_resid ? sr : sp;
    // run > u W  <=>  run > floor(u W) for the integer running weights
    const unsigned long long target =
        static_cast<unsigned long long>(static_cast<double>(sh.u_sample) * static_cast<double>(W));
    const unsigned long long base = use_resid ? br : bp, mine = use_resid ? cr : cp;
    const bool draws = (base <= target && target < base + mine) || (target >= W && rank == (use_resid ? lr : lp));
    if (draws) {
        const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
        unsigned long long incl = own;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off)
                incl += y;
        }
        __syncthreads();
        if (lane == 31)
            sh.ured[wid] = incl;
        __syncthreads();
        unsigned long long wbase = base;
        for (int i = 0; i < wid; ++i)
            wbase += sh.ured[i];
        const unsigned long long excl = wbase + incl - own;
        if (threadIdx.x == 0)
            sh.ired[0] = -1;
        __syncthreads();
        if (excl <= target && target < excl + own) {  // exactly one thread: the run of the draw
            unsigned long long run = excl;
            for (int c = c0, found = 0; c < c1 && !found; ++c) {
                float xp[8], xq[8];
                const int n = load_chunk(a, prow, c, xp);
                if (use_resid)
                    load_chunk(a, qrow, c, xq);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < n && !found) {
                        run += use_resid ? wr_of(xp[i], xq[i]) : wp_of(xp[i]);
                        if (run > target) {
                            sh.ired[0] = c * per + i;
                            found = 1;
                        }
                    }
            }
        }
        __syncthreads();
        int token = sh.ired[0];
        if (token < 0) {  // target rounded up to the total: the last token with weight
            int haswt = -1;
            if (own > 0)
                for (int c = c1 - 1; c >= c0 && haswt < 0; --c) {
                    float xp[8], xq[8];
                    const int n = load_chunk(a, prow, c, xp);
                    if (use_resid)
                        load_chunk(a, qrow, c, xq);
#pragma unroll
                    for (int i = 7; i >= 0; --i)
                        if (i < n && haswt < 0 && (use_resid ? wr_of(xp[i], xq[i]) : wp_of(xp[i])) > 0)
                            haswt = c * per + i;
                }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                haswt = max(haswt, __shfl_xor_sync(0xffffffffu, haswt, off));
            if (lane == 0)
                sh.ired2[wid] = haswt;
            __syncthreads();
            for (int i = 0; i < SNW; ++i)
                token = max(token, sh.ired2[i]);
        }
        if (threadIdx.x == 0)
            finish(token);
    }
    if (CL > 1)
        cluster_wait();  // no CTA leaves while another may still read its parts
}

// One CTA a session.
__global__ void __launch_bounds__(SNT) walk_kernel(const SampArgs a, const RowStats *__restrict__ stats)
{
    __shared__ WalkShared sh;
    walk_session<1>(sh, a, stats, blockIdx.x);
}

// A cluster of CL CTAs a session (few sessions: one CTA would weight the whole row).
template <int CL>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(SNT, 1)
    walk_cluster_kernel(const SampArgs a, const RowStats *__restrict__ stats)
{
    __shared__ WalkShared sh;
    walk_session<CL>(sh, a, stats, blockIdx.x / CL);
}

int check_sampling(const kda_sampling *sp)
{
    if (!sp)
        return fail(KDA_EINVAL, "sampling parameters must not be NULL");
    if (!(sp->temperature > 0.f) || !(sp->temperature < INFINITY))
        return fail(KDA_EINVAL, "temperature must be positive and finite");
    if (sp->top_k < 0)
        return fail(KDA_EINVAL, "top_k must be >= 0 (0: off; >= V keeps every token)");
    if (!(sp->top_p > 0.f) || sp->top_p > 1.f)
        return fail(KDA_EINVAL, "top_p must lie in (0, 1]");
    if (!(sp->min_p >= 0.f) || !(sp->min_p < 1.f))
        return fail(KDA_EINVAL, "min_p must lie in [0, 1)");
    return KDA_OK;
}

// Once per device (under a lock): the SM count, and the row-statistics launches' dynamic
// shared memory above the default 48 KiB.
int device_setup(int &sms)
{
    struct Info {
        std::atomic<int> ready{0};
        int sms = 0;
    };
    static Info info[64];
    static std::mutex init_mutex;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(KDA_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64)
        return fail(KDA_EINVAL, "device ordinal beyond the launch table");
    Info &di = info[dev];
    if (!di.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(init_mutex);
        if (!di.ready.load(std::memory_order_relaxed)) {
            int n = 0;
            e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
            const void *kernels[4] = {reinterpret_cast<const void *>(row_stats_kernel),
                                      reinterpret_cast<const void *>(row_stats_cluster_kernel<8>),
                                      reinterpret_cast<const void *>(row_stats_cluster_kernel<4>),
                                      reinterpret_cast<const void *>(row_stats_cluster_kernel<2>)};
            for (const void *k : kernels)
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(ROW_SMEM));
            if (e != cudaSuccess)
                return fail(KDA_ECUDA, std::string("sampled accept set-up: ") + cudaGetErrorString(e));
            di.sms = n;
            di.ready.store(1, std::memory_order_release);
        }
    }
    sms = di.sms;
    return KDA_OK;
}

// Shared body of both entry points: u_accept/u_sample or seeds/counters.
int sampled_common(const void *logits, const void *draft_logits, int logit_dtype, int B, int T, int V,
                   const int *drafts, const float *u_accept, const float *u_sample, const unsigned long long *seeds,
                   unsigned *counters, const kda_sampling *sp, int *j_out, int *token_out, int *keep_out,
                   int *dev_status, void *scratch, size_t scratch_bytes, cudaStream_t stream)
{
    if (B < 0)
        return fail(KDA_EINVAL, "B must be >= 0");
    if (T < 1 || T > KDA_TMAX)
        return fail(KDA_EINVAL, "T must lie in 1..15, got " + std::to_string(T));
    if (V < 1 || V > KDA_SAMPLED_VMAX)
        return fail(KDA_EINVAL, "V must lie in 1.." + std::to_string(KDA_SAMPLED_VMAX) +
                                    " (the fixed-point sums of the weights hold 2^64 / 2^46 of them)");
    if (logit_dtype != KDA_F32 && logit_dtype != KDA_BF16)
        return fail(KDA_EINVAL, "logit_dtype must be KDA_F32 or KDA_BF16");
    int rc = check_sampling(sp);
    if (rc)
        return rc;
    if (B == 0)
        return ok();
    const bool session = seeds != nullptr;
    if (!logits || !j_out || !token_out || (T > 1 && (!draft_logits || !drafts)))
        return fail(KDA_EINVAL, "logits, draft_logits, drafts, j_out and token_out must not be NULL");
    if (session ? !counters : (!u_sample || (T > 1 && !u_accept)))
        return fail(KDA_EINVAL, session ? "counters must not be NULL" : "u_accept and u_sample must not be NULL");
    if (session && ((reinterpret_cast<uintptr_t>(seeds) & 7u) || (reinterpret_cast<uintptr_t>(counters) & 7u)))
        return fail(KDA_EINVAL, "seeds and counters must be 8-byte aligned");
    const uintptr_t al = logit_dtype == KDA_BF16 ? 1u : 3u;
    if ((reinterpret_cast<uintptr_t>(logits) & al) || (reinterpret_cast<uintptr_t>(draft_logits) & al))
        return fail(KDA_EINVAL, "logits must be aligned to their element type");
    const size_t need = static_cast<size_t>(B) * (2 * T - 1) * sizeof(RowStats);
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
    a.seeds = seeds;
    a.counters = counters;
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
    const long long rows = static_cast<long long>(B) * (2 * T - 1);
    int sms = 0;
    if ((rc = device_setup(sms)))
        return rc;
    // few rows: a cluster of CTAs a row, as many as keep every cluster resident at once
    // (one CTA an SM); more rows than that keep one CTA a row (measured on GB300 at
    // V = 32768: 60 rows in three waves of 8-CTA clusters ran 94.8 -> 140 us)
    const unsigned gr = static_cast<unsigned>(rows);
    if (rows * 8 <= sms)
        row_stats_cluster_kernel<8><<<gr * 8, SNT, ROW_SMEM, stream>>>(a, stats);
    else if (rows * 4 <= sms)
        row_stats_cluster_kernel<4><<<gr * 4, SNT, ROW_SMEM, stream>>>(a, stats);
    else if (rows * 2 <= sms)
        row_stats_cluster_kernel<2><<<gr * 2, SNT, ROW_SMEM, stream>>>(a, stats);
    else
        row_stats_kernel<<<gr, SNT, ROW_SMEM, stream>>>(a, stats);
    if ((rc = check_launch("row statistics")))
        return rc;
    // the walk: a cluster of 8, 4 or 2 CTAs a session while the clusters fit on the GPU at
    // once, else one CTA a session
    const long long bs = B;
    const unsigned gb = static_cast<unsigned>(B);
    if (bs * 8 <= sms)
        walk_cluster_kernel<8><<<gb * 8, SNT, 0, stream>>>(a, stats);
    else if (bs * 4 <= sms)
        walk_cluster_kernel<4><<<gb * 4, SNT, 0, stream>>>(a, stats);
    else if (bs * 2 <= sms)
        walk_cluster_kernel<2><<<gb * 2, SNT, 0, stream>>>(a, stats);
    else
        walk_kernel<<<B, SNT, 0, stream>>>(a, stats);
    return check_launch("walk");
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
    return sampled_common(logits, draft_logits, logit_dtype, B, T, V, drafts, u_accept, u_sample, nullptr, nullptr,
                          sp, j_out, token_out, keep_out, dev_status, scratch, scratch_bytes, stream);
}

extern "C" int spec_accept_sampled_session(const void *logits, const void *draft_logits, int logit_dtype, int B,
                                           int T, int V, const int *drafts, const unsigned long long *seeds,
                                           unsigned *counters, const kda_sampling *sp, int *j_out, int *token_out,
                                           int *keep_out, int *dev_status, void *scratch, size_t scratch_bytes,
                                           cudaStream_t stream)
{
    if (B > 0 && !seeds)
        return fail(KDA_EINVAL, "seeds must not be NULL");
    return sampled_common(logits, draft_logits, logit_dtype, B, T, V, drafts, nullptr, nullptr, seeds, counters, sp,
                          j_out, token_out, keep_out, dev_status, scratch, scratch_bytes, stream);
}

extern "C" int kda_philox4x32_10(const unsigned *ctr, const unsigned *key, unsigned *out, int n, cudaStream_t stream)
{
    if (n < 0)
        return fail(KDA_EINVAL, "n must be >= 0");
    if (n == 0)
        return ok();
    if (!ctr || !key || !out)
        return fail(KDA_EINVAL, "ctr, key and out must not be NULL");
    if (!aligned16(ctr) || !aligned16(out) || (reinterpret_cast<uintptr_t>(key) & 7u))
        return fail(KDA_EINVAL, "ctr and out must be 16-byte aligned, key 8-byte aligned");
    const int grid = static_cast<int>(std::min<long long>((n + 255) / 256, 4096));
    philox_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint4 *>(ctr), reinterpret_cast<const uint2 *>(key),
                                            reinterpret_cast<uint4 *>(out), n);
    return check_launch("philox_kernel");
}
