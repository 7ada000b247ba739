// spec_accept.cu -- greedy acceptance over the verify logits (sm_103a).
//
// glm_spec.rs (memra-engine 0.123.0), glm5_spec_round step 4: one device argmax
// per verify row with the lowest index winning ties, one small readback, then
// j = the first row whose draft differs from the row's argmax (else K) and the
// bonus token vam[j]; keep = j + 1 (the anchor row is always committed).  A row
// holding a NaN has no argmax; reaching it refuses loudly (guard_vocab_token).
//
// spec_accept and spec_accept_var: one launch of thread-block clusters, one cluster
// of CL CTAs per session.  CTA c of a cluster reduces vocabulary slice c of every
// row of the session (warp w takes rows w, w + 8) to (max, lowest index of the max,
// NaN seen) and writes that triple into the shared memory of the cluster's first
// CTA (distributed shared memory); after the cluster barrier, lane r of that CTA's
// first warp folds the CL triples of row r in slice order, and a ballot over the
// mismatch predicate gives j.
// spec_accept_noalloc keeps the two-launch form, whose partial results go through a
// scratch array:
//   1. accept_partial_kernel: grid (B*T rows, VS slices of the vocabulary); each
//      CTA reduces its slice to the triple and writes it to scratch.
//   2. accept_final_kernel: one warp per session folds the VS triples of each row.
// The selection is a total order on (value, -index), so the reduction order
// never changes the result.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int ACC_THREADS = 256;
constexpr int SLICE = 4096;  // logits per CTA of the first pass
constexpr int MAX_VS = 64;

struct Partial {
    float v;
    int idx;
    int nan;
    int pad;
};

__host__ __device__ inline int slices_for(int V)
{
    int vs = (V + SLICE - 1) / SLICE;
    return vs < 1 ? 1 : (vs > MAX_VS ? MAX_VS : vs);
}

__device__ __forceinline__ void take(float &bv, int &bi, float v, int i)
{
    if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
    }
}

template <bool BF16>
__global__ void __launch_bounds__(ACC_THREADS) accept_partial_kernel(const void *__restrict__ logits, int V,
                                                                      int vs, int chunk, Partial *__restrict__ part,
                                                                      const int *__restrict__ t_rows, int T)
{
    const long long row = blockIdx.x;
    const int s = blockIdx.y;
    // with per-session row counts, rows past a session's count are never consulted
    if (t_rows && static_cast<int>(row % T) >= t_rows[row / T])
        return;
    const int begin = s * chunk;
    const int end = min(V, begin + chunk);
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    int nan = 0;
    if (BF16) {
        const uint16_t *x = static_cast<const uint16_t *>(logits) + row * V;
        const bool vec = (V % 8 == 0) && (chunk % 8 == 0);
        if (vec) {
            const uint4 *x8 = reinterpret_cast<const uint4 *>(x);
            for (int c8 = begin / 8 + threadIdx.x; c8 < end / 8; c8 += ACC_THREADS) {
                const uint4 r = x8[c8];
                const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float lo = __uint_as_float(w[m] << 16), hi = __uint_as_float(w[m] & 0xffff0000u);
                    nan |= (lo != lo) | (hi != hi);
                    take(bv, bi, lo, 8 * c8 + 2 * m);
                    take(bv, bi, hi, 8 * c8 + 2 * m + 1);
                }
            }
        } else {
            for (int c = begin + threadIdx.x; c < end; c += ACC_THREADS) {
                const float v = __uint_as_float(static_cast<uint32_t>(x[c]) << 16);
                nan |= (v != v);
                take(bv, bi, v, c);
            }
        }
    } else {
        const float *x = static_cast<const float *>(logits) + row * V;
        const bool vec = (V % 4 == 0) && (chunk % 4 == 0);
        if (vec) {
            const float4 *x4 = reinterpret_cast<const float4 *>(x);
            for (int c4 = begin / 4 + threadIdx.x; c4 < end / 4; c4 += ACC_THREADS) {
                const float4 r = x4[c4];
                nan |= (r.x != r.x) | (r.y != r.y) | (r.z != r.z) | (r.w != r.w);
                take(bv, bi, r.x, 4 * c4);
                take(bv, bi, r.y, 4 * c4 + 1);
                take(bv, bi, r.z, 4 * c4 + 2);
                take(bv, bi, r.w, 4 * c4 + 3);
            }
        } else {
            for (int c = begin + threadIdx.x; c < end; c += ACC_THREADS) {
                const float v = x[c];
                nan |= (v != v);
                take(bv, bi, v, c);
            }
        }
    }
    // NaN never wins `take` (every comparison with NaN is false)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        nan |= __shfl_xor_sync(0xffffffffu, nan, off);
        take(bv, bi, ov, oi);
    }
    __shared__ float sv[ACC_THREADS / 32];
    __shared__ int si[ACC_THREADS / 32], sn[ACC_THREADS / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (lane == 0) {
        sv[wid] = bv;
        si[wid] = bi;
        sn[wid] = nan;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < ACC_THREADS / 32; ++w) {
            take(bv, bi, sv[w], si[w]);
            nan |= sn[w];
        }
        Partial pt;
        pt.v = bv;
        pt.idx = bi;
        pt.nan = nan;
        pt.pad = 0;
        part[row * vs + s] = pt;
    }
}

// t_rows (nullable): session b's round has t_rows[b] rows of the T in the layout; its
// drafts are drafts[b][0 .. t_rows[b]-2] (the layout keeps T-1 draft slots per session).
__global__ void accept_final_kernel(const Partial *__restrict__ part, int B, int T, int vs,
                                    const int *__restrict__ drafts, int *j_out, int *bonus_out, int *keep_out,
                                    int *status, const int *__restrict__ t_rows)
{
    const int warps = blockDim.x / 32;
    const int b = blockIdx.x * warps + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (b >= B)
        return;
    const int Tb = t_rows ? t_rows[b] : T;
    if (Tb < 1 || Tb > T) {  // an invalid row count: no accept for this session
        if (lane == 0) {
            if (j_out)
                j_out[b] = -1;
            if (bonus_out)
                bonus_out[b] = -1;
            if (keep_out)
                keep_out[b] = 0;
            if (status)
                atomicOr(status, KDA_ST_BADKEEP);
        }
        return;
    }
    const int K = Tb - 1;
    int vam = -1;
    if (lane < Tb) {
        const Partial *pr = part + (static_cast<long long>(b) * T + lane) * vs;
        float bv = -INFINITY;
        int bi = 0x7fffffff, nan = 0;
        for (int s = 0; s < vs; ++s) {
            const Partial q = pr[s];
            nan |= q.nan;
            take(bv, bi, q.v, q.idx);
        }
        vam = nan ? -1 : bi;
    }
    const bool miss = lane < K && (vam < 0 || drafts[static_cast<long long>(b) * (T - 1) + lane] != vam);
    const unsigned mask = __ballot_sync(0xffffffffu, miss);
    const int j = mask ? __ffs(mask) - 1 : K;
    const int bonus = __shfl_sync(0xffffffffu, vam, j);
    if (lane == 0) {
        if (j_out)
            j_out[b] = j;
        if (bonus_out)
            bonus_out[b] = bonus;
        if (keep_out)
            keep_out[b] = j + 1;
        if (bonus < 0 && status)
            atomicOr(status, KDA_ST_NAN);
    }
}

constexpr int CL = 8;  // CTAs (vocabulary slices) per session: one cluster

// The (max, lowest index, NaN seen) triple of logits [begin, end) of one row, reduced
// over a warp (every lane ends with the triple).  A lane issues up to NB 16-byte loads
// before it compares any of them, so a slice costs one load latency, not NB.
constexpr int NB = 16;

template <bool BF16>
__device__ __forceinline__ Partial warp_slice(const void *logits, long long row, int V, int begin, int end, int lane)
{
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    int nan = 0;
    constexpr int PER = BF16 ? 8 : 4;  // logits per 16-byte vector
    const char *x = static_cast<const char *>(logits) + row * V * (BF16 ? 2 : 4);
    if (V % PER == 0 && begin % PER == 0 && end % PER == 0) {
        const uint4 *xv = reinterpret_cast<const uint4 *>(x);
        for (int c0 = begin / PER; c0 < end / PER; c0 += 32 * NB) {
            uint4 r[NB];
#pragma unroll
            for (int i = 0; i < NB; ++i) {
                const int c = c0 + lane + 32 * i;
                r[i] = c < end / PER ? xv[c] : make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu);
            }
#pragma unroll
            for (int i = 0; i < NB; ++i) {
                const int c = c0 + lane + 32 * i;
                if (c >= end / PER)
                    break;
                const uint32_t w[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
                if (BF16) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float lo = __uint_as_float(w[m] << 16), hi = __uint_as_float(w[m] & 0xffff0000u);
                        nan |= (lo != lo) | (hi != hi);
                        take(bv, bi, lo, 8 * c + 2 * m);
                        take(bv, bi, hi, 8 * c + 2 * m + 1);
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float v = __uint_as_float(w[m]);
                        nan |= (v != v);
                        take(bv, bi, v, 4 * c + m);
                    }
                }
            }
        }
    } else {
        for (int c = begin + lane; c < end; c += 32) {
            const float v = BF16 ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(x)[c]) << 16)
                                 : reinterpret_cast<const float *>(x)[c];
            nan |= (v != v);
            take(bv, bi, v, c);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        nan |= __shfl_xor_sync(0xffffffffu, nan, off);
        take(bv, bi, ov, oi);
    }
    return Partial{bv, bi, nan, 0};
}

// grid B * CL CTAs of ACC_THREADS, clusters of CL; chunk: logits per slice (a multiple
// of 8).  t_rows (nullable) as for accept_final_kernel.
template <bool BF16>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(ACC_THREADS)
    accept_cluster_kernel(const void *__restrict__ logits, int V, int T, int chunk, const int *__restrict__ drafts,
                          int *j_out, int *bonus_out, int *keep_out, int *status, const int *__restrict__ t_rows)
{
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ Partial part[KDA_TMAX][CL];  // in the first CTA: every slice's triple of every row
    asm volatile("griddepcontrol.wait;" ::: "memory");  // launched as a programmatic dependent
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int rank = static_cast<int>(cluster.block_rank());
    const int b = blockIdx.x / CL;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int Tb = t_rows ? t_rows[b] : T;
    const bool valid = Tb >= 1 && Tb <= T;
    const int begin = min(V, rank * chunk), end = min(V, begin + chunk);
    Partial *lead = cluster.map_shared_rank(&part[0][0], 0);
    if (valid) {
        // rows past a session's count are never consulted
        for (int r = wid; r < Tb; r += ACC_THREADS / 32) {
            const Partial pt = BF16 ? warp_slice<true>(logits, static_cast<long long>(b) * T + r, V, begin, end, lane)
                                    : warp_slice<false>(logits, static_cast<long long>(b) * T + r, V, begin, end, lane);
            if (lane == 0)
                lead[r * CL + rank] = pt;
        }
    }
    cluster.sync();  // every slice's triples are in the first CTA's shared memory
    if (rank != 0 || wid != 0)
        return;
    if (!valid) {  // an invalid row count: no accept for this session
        if (lane == 0) {
            if (j_out)
                j_out[b] = -1;
            if (bonus_out)
                bonus_out[b] = -1;
            if (keep_out)
                keep_out[b] = 0;
            if (status)
                atomicOr(status, KDA_ST_BADKEEP);
        }
        return;
    }
    const int K = Tb - 1;
    int vam = -1;
    if (lane < Tb) {
        float bv = -INFINITY;
        int bi = 0x7fffffff, nan = 0;
        for (int c = 0; c < CL; ++c) {
            const Partial q = part[lane][c];
            nan |= q.nan;
            take(bv, bi, q.v, q.idx);
        }
        vam = nan ? -1 : bi;
    }
    const bool miss = lane < K && (vam < 0 || drafts[static_cast<long long>(b) * (T - 1) + lane] != vam);
    const unsigned mask = __ballot_sync(0xffffffffu, miss);
    const int j = mask ? __ffs(mask) - 1 : K;
    const int bonus = __shfl_sync(0xffffffffu, vam, j);
    if (lane == 0) {
        if (j_out)
            j_out[b] = j;
        if (bonus_out)
            bonus_out[b] = bonus;
        if (keep_out)
            keep_out[b] = j + 1;
        if (bonus < 0 && status)
            atomicOr(status, KDA_ST_NAN);
    }
}

// One cluster launch for B sessions.
int launch_accept_cluster(const void *logits, int logit_dtype, int B, int T, int V, const int *drafts, int *j_out,
                          int *bonus_out, int *keep_out, int *dev_status, const int *t_rows, cudaStream_t stream)
{
    if (static_cast<long long>(B) * CL > 0x7fffffffLL)
        return fail(KDA_EINVAL, "B exceeds the grid limit");
    int chunk = (V + CL - 1) / CL;
    chunk = (chunk + 7) / 8 * 8;
    const unsigned grid = static_cast<unsigned>(B) * CL;
    // programmatic dependent launch, as the scan kernel: the kernel waits for the
    // previous kernel's results before it reads anything
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(ACC_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le =
        logit_dtype == KDA_BF16
            ? cudaLaunchKernelEx(&cfg, accept_cluster_kernel<true>, logits, V, T, chunk, drafts, j_out, bonus_out,
                                 keep_out, dev_status, t_rows)
            : cudaLaunchKernelEx(&cfg, accept_cluster_kernel<false>, logits, V, T, chunk, drafts, j_out, bonus_out,
                                 keep_out, dev_status, t_rows);
    if (le != cudaSuccess)
        return fail(KDA_ECUDA, std::string("accept_cluster_kernel launch: ") + cudaGetErrorString(le));
    return check_launch("accept_cluster_kernel");
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" size_t spec_accept_scratch_bytes(int B, int T, int V)
{
    if (B <= 0 || T <= 0 || V <= 0)
        return 0;
    return static_cast<size_t>(B) * T * slices_for(V) * sizeof(Partial);
}

extern "C" int spec_accept(const void *logits, int logit_dtype, int B, int T, int V, const int *drafts,
                           int *j_out, int *bonus_out, int *keep_out, int *dev_status, void *scratch,
                           size_t scratch_bytes, cudaStream_t stream)
{
    if (B < 0)
        return fail(KDA_EINVAL, "B must be >= 0");
    if (T < 1 || T > KDA_TMAX)
        return fail(KDA_EINVAL, "T must lie in 1..15, got " + std::to_string(T));
    if (V < 1)
        return fail(KDA_EINVAL, "V must be >= 1");
    if (logit_dtype != KDA_F32 && logit_dtype != KDA_BF16)
        return fail(KDA_EINVAL, "logit_dtype must be KDA_F32 or KDA_BF16");
    if (B == 0)
        return ok();
    if (!logits || (T > 1 && !drafts))
        return fail(KDA_EINVAL, "logits and drafts must not be NULL");
    if (!aligned16(logits))
        return fail(KDA_EINVAL, "logits must be 16-byte aligned");
    // the cluster form passes its partial results through shared memory: the scratch
    // arguments stay in the signature for existing callers and are not used
    (void)scratch;
    (void)scratch_bytes;
    return launch_accept_cluster(logits, logit_dtype, B, T, V, drafts, j_out, bonus_out, keep_out, dev_status,
                                 nullptr, stream);
}

// ---------------------------------------------------------------------------
// spec_accept_noalloc: the same two passes, with the per-slice partial results
// kept in a fixed array that lives in the library's device image instead of
// caller scratch.  For callers that cannot allocate device memory at the point
// where they accept a round (see the declaration in kda_spec.h).
// ---------------------------------------------------------------------------
#include <mutex>

namespace kda {
namespace {

constexpr size_t NOALLOC_SCRATCH = KDA_NOALLOC_SCRATCH_BYTES;
constexpr int MAX_DEVICES = 64;

// One copy per device that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char g_accept_scratch[NOALLOC_SCRATCH];

std::mutex g_scratch_mutex;
struct ScratchAddr {
    CUcontext ctx;  // the context the address was looked up in
    void *addr;
};
ScratchAddr g_scratch_addr[MAX_DEVICES] = {};

using CtxGetCurrent = PFN_cuCtxGetCurrent_v4000;

CtxGetCurrent lookup_ctx_get_current()
{
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<CtxGetCurrent>(f);
}

// Device address of g_accept_scratch on the current device.  On the host the
// symbol is only a stand-in, so its address is looked up with the device current
// and kept per device together with the context it belongs to; a call in another
// context (after cudaDeviceReset, say, or with a context of the caller's own) looks
// it up again.
int noalloc_scratch(void **addr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(KDA_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= MAX_DEVICES)
        return fail(KDA_EINVAL, "device ordinal beyond the no-allocation table");
    static const CtxGetCurrent ctx_get = lookup_ctx_get_current();
    if (!ctx_get)
        return fail(KDA_ECUDA, "cuCtxGetCurrent is not available from the CUDA driver");
    CUcontext ctx = nullptr;
    if (ctx_get(&ctx) != CUDA_SUCCESS)
        return fail(KDA_ECUDA, "cuCtxGetCurrent failed");
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchAddr &sa = g_scratch_addr[dev];
    if (!ctx || !sa.addr || sa.ctx != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_accept_scratch);  // makes the device's context current if none was
        if (e != cudaSuccess || !p)
            return fail(KDA_ECUDA, std::string("cudaGetSymbolAddress(accept scratch): ") + cudaGetErrorString(e));
        if (ctx_get(&ctx) != CUDA_SUCCESS || !ctx)
            return fail(KDA_ECUDA, "cuCtxGetCurrent failed");
        sa.ctx = ctx;
        sa.addr = p;
    }
    *addr = sa.addr;
    return KDA_OK;
}

}  // namespace
}  // namespace kda

extern "C" int spec_accept_noalloc(const void *logits, int logit_dtype, int B, int T, int V, const int *drafts,
                                   int *j_out, int *bonus_out, int *keep_out, int *dev_status, cudaStream_t stream)
{
    if (B < 0)
        return fail(KDA_EINVAL, "B must be >= 0");
    if (T < 1 || T > KDA_TMAX)
        return fail(KDA_EINVAL, "T must lie in 1..15, got " + std::to_string(T));
    if (V < 1)
        return fail(KDA_EINVAL, "V must be >= 1");
    if (logit_dtype != KDA_F32 && logit_dtype != KDA_BF16)
        return fail(KDA_EINVAL, "logit_dtype must be KDA_F32 or KDA_BF16");
    if (B == 0)
        return ok();
    if (!logits || (T > 1 && !drafts))
        return fail(KDA_EINVAL, "logits and drafts must not be NULL");
    if (!aligned16(logits))
        return fail(KDA_EINVAL, "logits must be 16-byte aligned");
    const size_t need = spec_accept_scratch_bytes(B, T, V);
    if (need > NOALLOC_SCRATCH)
        return fail(KDA_EINVAL, "spec_accept_noalloc: B=" + std::to_string(B) + ", T=" + std::to_string(T) +
                                    ", V=" + std::to_string(V) + " needs " + std::to_string(need) +
                                    " bytes of scratch, above its fixed " + std::to_string(NOALLOC_SCRATCH) +
                                    "; call spec_accept with caller scratch instead");
    void *scratch = nullptr;
    int rc = noalloc_scratch(&scratch);
    if (rc)
        return rc;
    const int vs = slices_for(V);
    int chunk = (V + vs - 1) / vs;
    chunk = (chunk + 7) / 8 * 8;
    Partial *part = static_cast<Partial *>(scratch);
    dim3 grid(static_cast<unsigned>(B * T), static_cast<unsigned>(vs));
    if (logit_dtype == KDA_BF16)
        accept_partial_kernel<true><<<grid, ACC_THREADS, 0, stream>>>(logits, V, vs, chunk, part, nullptr, T);
    else
        accept_partial_kernel<false><<<grid, ACC_THREADS, 0, stream>>>(logits, V, vs, chunk, part, nullptr, T);
    rc = check_launch("accept_partial_kernel");
    if (rc)
        return rc;
    const int warps = 4;
    accept_final_kernel<<<(B + warps - 1) / warps, warps * 32, 0, stream>>>(part, B, T, vs, drafts, j_out,
                                                                            bonus_out, keep_out, dev_status, nullptr);
    return check_launch("accept_final_kernel");
}

// ---------------------------------------------------------------------------
// Per-session round lengths: spec_accept_var (greedy accept when session b ran
// t_rows[b] of the T rows) and spec_window (the verify-window policies that pick
// t_rows from the drafter's slot scores).
// ---------------------------------------------------------------------------
namespace kda {
namespace {

__device__ __forceinline__ float sigmoid_ieee(float r)
{
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-r)));
}

// One thread per session: scores [B][K]; writes t_out[b] = the session's verify rows.
//   KDA_WIN_CONF_KEEP        glm_spec.rs glm5_conf_keep: scores are slot confidences q,
//                            param = p_min, pmin0 arms the slot-0 break; rows = 1 + kept.
//   KDA_WIN_CONFIDENCE       dflash.rs dspark_confidence_vt: scores are pre-sigmoid raws,
//                            param = tau, cumulative survival; rows in [2, max(t_cap, 2)].
//   KDA_WIN_SLOT_CONFIDENCE  dflash.rs dspark_slot_confidence_vt: per-slot sigmoid >= tau.
// Every result is capped at t_cap.
__global__ void window_kernel(const float *__restrict__ scores, int B, int K, int policy, float param, int pmin0,
                              int t_cap, int *__restrict__ t_out)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B)
        return;
    const float *x = scores + static_cast<long long>(b) * K;
    int kept = 0;
    if (policy == KDA_WIN_CONF_KEEP) {
        for (int j = 0; j < K; ++j) {
            if (x[j] < param && (j > 0 || pmin0))
                break;
            ++kept;
        }
        t_out[b] = min(1 + kept, t_cap);
        return;
    }
    float surv = 1.0f;
    for (int k = 0; k < K; ++k) {
        const float sg = sigmoid_ieee(x[k]);
        if (policy == KDA_WIN_CONFIDENCE) {
            surv = __fmul_rn(surv, sg);
            if (surv < param)
                break;
        } else if (sg < param) {
            break;
        }
        ++kept;
    }
    const int hi = t_cap > 2 ? t_cap : 2;
    t_out[b] = min(max(1 + kept, 2), hi);
}

}  // namespace
}  // namespace kda

extern "C" int spec_accept_var(const void *logits, int logit_dtype, int B, int T, int V, const int *t_rows,
                               const int *drafts, int *j_out, int *bonus_out, int *keep_out, int *dev_status,
                               void *scratch, size_t scratch_bytes, cudaStream_t stream)
{
    if (B < 0)
        return fail(KDA_EINVAL, "B must be >= 0");
    if (T < 1 || T > KDA_TMAX)
        return fail(KDA_EINVAL, "T must lie in 1..15, got " + std::to_string(T));
    if (V < 1)
        return fail(KDA_EINVAL, "V must be >= 1");
    if (logit_dtype != KDA_F32 && logit_dtype != KDA_BF16)
        return fail(KDA_EINVAL, "logit_dtype must be KDA_F32 or KDA_BF16");
    if (B == 0)
        return ok();
    if (!logits || !t_rows || (T > 1 && !drafts))
        return fail(KDA_EINVAL, "logits, t_rows and drafts must not be NULL");
    if (!aligned16(logits) || (reinterpret_cast<uintptr_t>(t_rows) & 3u))
        return fail(KDA_EINVAL, "logits must be 16-byte and t_rows 4-byte aligned");
    (void)scratch;  // not used by the cluster form, as in spec_accept
    (void)scratch_bytes;
    return launch_accept_cluster(logits, logit_dtype, B, T, V, drafts, j_out, bonus_out, keep_out, dev_status,
                                 t_rows, stream);
}

extern "C" int spec_window(const float *scores, int B, int K, int policy, float param, int pmin0, int t_cap,
                           int *t_out, cudaStream_t stream)
{
    if (B < 0 || K < 0)
        return fail(KDA_EINVAL, "B and K must be >= 0");
    if (policy != KDA_WIN_CONF_KEEP && policy != KDA_WIN_CONFIDENCE && policy != KDA_WIN_SLOT_CONFIDENCE)
        return fail(KDA_EINVAL, "policy must be KDA_WIN_CONF_KEEP, KDA_WIN_CONFIDENCE or KDA_WIN_SLOT_CONFIDENCE");
    const int lo = policy == KDA_WIN_CONF_KEEP ? 1 : 2;
    if (t_cap < lo || t_cap > KDA_TMAX)
        return fail(KDA_EINVAL, "t_cap must lie in " + std::to_string(lo) + "..15 for this policy, got " +
                                    std::to_string(t_cap));
    if (!(param == param))
        return fail(KDA_EINVAL, "param must not be NaN");
    if (B == 0)
        return ok();
    if ((K > 0 && !scores) || !t_out)
        return fail(KDA_EINVAL, "scores and t_out must not be NULL");
    if ((reinterpret_cast<uintptr_t>(scores) & 3u) || (reinterpret_cast<uintptr_t>(t_out) & 3u))
        return fail(KDA_EINVAL, "scores and t_out must be 4-byte aligned");
    const int threads = 128;
    window_kernel<<<(B + threads - 1) / threads, threads, 0, stream>>>(scores, B, K, policy, param, pmin0, t_cap,
                                                                       t_out);
    return check_launch("window_kernel");
}
