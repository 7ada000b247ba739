// kda_scan.cu -- the fused KDA verify walk (short conv, activations, gated delta
// rule) for sm_103a, and the accept-j rollback that replays it.
//
// One persistent kernel serves both.  A unit is one (layer, session, head): its
// 128 x 128 f32 state, the raw rows of its T drafted positions, its conv ring and
// conv weights.  Each CTA (8 warps, 2 per SM) walks units blockIdx.x, +gridDim.x,
// ... and keeps one unit's state in registers for its whole T-row loop, so the 64
// KiB state of a head crosses HBM once in and once out per round.
//
// Memory pipeline per CTA (bulk copies = the 1D TMA, counted by mbarriers):
//   - the next unit's raw rows, ring and weights are bulk-loaded into a stage as
//     soon as the current unit's prologue has consumed them;
//   - the current unit's pre-round state leaves the stage as a bulk store to the
//     snapshot (the fused snapshot write) while the unit scans, after which the
//     next unit's state is bulk-loaded into the stage;
//   - the scanned state is stored from registers.
// Every wait on an mbarrier is bounded; a wait that runs out sets KDA_ST_TIMEOUT,
// lets the copies in flight land and ends the CTA.
//
// Register tile: lane 4 rg + cg of warp wi holds key rows 16 rg .. 16 rg + 15 of
// value columns 16 wi + 4 cg .. +3, with row pairs packed into float2 so each
// element operation is one lane of a packed f32x2 instruction (__fmul2_rn,
// __ffma2_rn).  Per row t (glm_spec.rs module doc, VERIFY-ROW BATCHING: the
// recurrence stays sequential inside one launch, the in-kernel T-loop being the
// chained t=1 program):
//   S' = d_t (.) S               d = exp(g), g = -5 sigmoid(raw_g)
//   u  = S'^T k,  e = S'^T q     one register sweep, then a 3-step shuffle
//                                reduce-scatter over the 8 row groups
//   w  = beta (v - u)
//   o  = (e + w (k.q)) / sqrt(128)   == (S' + k w^T)^T q / sqrt(128)
//   S  = S' + k w^T              second register sweep
// Every operation is an explicitly rounded intrinsic and the code for a row does
// not depend on T or on the unit, so T rows in one launch and T launches of one
// row give the same bits, and so do a rollback replay and a fresh verify.
//
// Prologue per unit: one warp per row computes the width-4 causal conv + SiLU of
// q, k, v (mini fixture linear_attn_config of glm5_spec_ppn_gate.rs:
// short_conv_kernel_size 4, head_dim 128, gate_lower_bound -5.0), the L2 norms
// of q and k, k.q, the gates and beta, with one fixed reduction tree per row,
// into shared memory that the T-loop reads as broadcast float4 loads.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <string>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int D = 128;
constexpr int NW = 8;           // warps per CTA
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

constexpr int MAX_POLLS = 1 << 24;  // mbarrier polls (with back-off, a few seconds) before giving up

// Shared memory of a CTA whose units run at most `tcap` rows; `es` is the raw-row
// element size.  The stage holds the NEXT unit's inputs, filled by bulk copies.
struct Layout {
    int tcap, es;
    __host__ __device__ size_t stage_state() const { return 0; }                       // [128][128] f32
    __host__ __device__ size_t stage_rows() const { return (size_t)D * D * 4; }         // [4: q,k,v,g][tcap][128]
    __host__ __device__ size_t stage_ring() const { return stage_rows() + (size_t)4 * tcap * D * es; }  // [3][3][128]
    __host__ __device__ size_t stage_w() const { return stage_ring() + (size_t)9 * D * 4; }   // [3][128] x 4 taps
    __host__ __device__ size_t vec() const { return stage_w() + (size_t)3 * D * 16; }         // [tcap][4][128] f32
    __host__ __device__ size_t beta() const { return vec() + (size_t)tcap * 4 * D * 4; }      // [16] f32
    __host__ __device__ size_t kq() const { return beta() + 64; }                             // [16] f32
    __host__ __device__ size_t bar() const { return kq() + 64; }  // mbarriers: [0] state stage, [1] the rest
    __host__ __device__ size_t total() const { return bar() + 16; }
};

// sigmoid through the fast exp2 / reciprocal intrinsics: relative error ~1e-6, far
// inside the 1e-4 parity bar, and a short dependency chain for the prologue
__device__ __forceinline__ float sigmoidf_(float z)
{
    return __fdividef(1.0f, __fadd_rn(1.0f, __expf(-z)));
}

__device__ __forceinline__ float load_scalar(const void *base, int bf16, size_t idx)
{
    if (bf16)
        return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t *>(base)[idx]) << 16);
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

// ---- bulk copies and the mbarrier that counts their bytes -------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// bulk store of shared memory to global memory, tracked by bulk groups
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// the bulk stores issued so far have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// the bulk stores issued so far are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait for the phase with `parity`; false after MAX_POLLS polls.
__device__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    for (int i = 0; i < MAX_POLLS; ++i) {
        if (mbar_try(bar, parity))
            return true;
        if (i >= 1024)
            __nanosleep(64);
    }
    return false;
}

// ---- units --------------------------------------------------------------------
struct Unit {
    int h, b, l, T;
    long long lb;  // l * B + b
};

// rows unit u runs: > 0 to run, 0 nothing to do, -1 an invalid device keep
__device__ __forceinline__ int unit_rows(const ScanParams &p, int b)
{
    if (p.keep_mode == KEEP_HOST) {
        const int kp = p.keep_host[b];  // validated 1..T_rows on the host
        return kp >= p.T_rows ? 0 : kp;
    }
    if (p.keep_mode == KEEP_DEVICE) {
        const int kp = p.keep_dev[b];
        if (kp < 1 || kp > p.T_rows)
            return -1;
        return kp == p.T_rows ? 0 : kp;
    }
    return p.T_run;
}

__device__ __forceinline__ Unit unit_of(const ScanParams &p, int u)
{
    Unit x;
    x.h = static_cast<int>(u % p.H);
    x.lb = u / p.H;
    x.b = static_cast<int>(x.lb % p.B);
    x.l = static_cast<int>(x.lb / p.B);
    x.T = unit_rows(p, x.b);
    return x;
}

// the first unit at or after u (stepping by the grid) that has rows to run
__device__ int next_live(const ScanParams &p, int u, int n)
{
    for (; u < n; u += gridDim.x) {
        const int T = unit_rows(p, static_cast<int>((u / p.H) % p.B));
        if (T > 0)
            return u;
        if (T < 0 && p.status && threadIdx.x == 0)
            atomicOr(p.status, KDA_ST_BADKEEP);  // the session is left untouched
    }
    return n;
}

// One thread fills the state stage with unit u's 64 KiB state.
__device__ void prefetch_state(const ScanParams &p, const Layout &lay, unsigned char *smem, uint32_t bar,
                               int u)
{
    mbar_expect_tx(bar, D * D * 4);
    for (int c = 0; c < 4; ++c)
        bulk_load(smem_addr(smem + lay.stage_state() + c * 16384), p.s_in + static_cast<size_t>(u) * D * D + c * 4096,
                  16384, bar);
}

// All threads fill the rest of the stage with unit u's raw rows (16-byte cp.async,
// spread over the CTA) and thread 32 adds the ring and conv weights as two bulk
// copies.  The input mbarrier completes once every thread's cp.async has landed
// (NT no-increment arrivals) and the bulk bytes have arrived (one expect_tx arrival).
__device__ void prefetch_inputs(const ScanParams &p, const Layout &lay, unsigned char *smem, uint32_t bar,
                                int u, int tid)
{
    const Unit x = unit_of(p, u);
    const int rbytes = D * lay.es, cpr = rbytes / 16, per_stream = x.T * cpr;
    const void *xs[4] = {p.xq, p.xk, p.xv, p.xg};
    for (int c = tid; c < 4 * per_stream; c += NT) {
        const int s = c / per_stream, rem = c - s * per_stream, t = rem / cpr, q = rem - t * cpr;
        const char *src = static_cast<const char *>(xs[s]) +
                          ((static_cast<size_t>(x.lb) * p.T_rows + t) * p.H + x.h) * static_cast<size_t>(rbytes) + 16 * q;
        const uint32_t dst = smem_addr(smem + lay.stage_rows() + static_cast<size_t>(s * lay.tcap + t) * rbytes + 16 * q);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
    }
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
    if (tid == 32) {  // not thread 0, which tends the state stage
        fence_proxy_async();  // the prologue's generic reads of the stage come first
        mbar_expect_tx(bar, 9 * D * 4 + 3 * D * 16);
        bulk_load(smem_addr(smem + lay.stage_ring()), p.ring_in + static_cast<size_t>(u) * 9 * D, 9 * D * 4, bar);
        bulk_load(smem_addr(smem + lay.stage_w()), p.conv_w + (static_cast<size_t>(x.l) * p.H + x.h) * 3 * D * 4,
                  3 * D * 16, bar);
    }
}

// four consecutive channels of stream s at extended index n (0..2 ring slots, 3+t row t)
__device__ __forceinline__ float4 fetch4(const Layout &lay, const unsigned char *smem, int s, int n, int c0)
{
    if (n < 3)
        return *reinterpret_cast<const float4 *>(smem + lay.stage_ring() + ((s * 3 + n) * D + c0) * 4);
    const unsigned char *r = smem + lay.stage_rows() + (static_cast<size_t>(s * lay.tcap + n - 3) * D + c0) * lay.es;
    if (lay.es == 4)
        return *reinterpret_cast<const float4 *>(r);
    const uint2 v = *reinterpret_cast<const uint2 *>(r);
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                       __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
}

// Persistent: each CTA walks units blockIdx.x, +gridDim.x, ...; while it scans
// one unit out of registers, the copies of its next unit are in flight.
__global__ void __launch_bounds__(NT, 2) kda_scan_kernel(const __grid_constant__ ScanParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const Layout lay{p.keep_mode == KEEP_NONE ? p.T_run : p.T_rows, p.bf16 ? 2 : 4};
    // thread (warp wi, lane = 4 rg + cg) holds key rows i = 16 rg + r (r < 16) of value
    // columns j = 16 wi + 4 cg + c (c < 4): 64 elements, row pairs packed as float2.
    // The 8 lanes of one cg (rg = 0..7) together cover all 128 rows of their 4 columns.
    const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5, cg = lane & 3, rg = lane >> 2;
    const int jbase = wi * 16 + 4 * cg;
    // after the reduce-scatter a lane holds one sum: of u (rg < 4) or e (rg >= 4), column jbase + (rg & 3)
    const int jsum = jbase + (rg & 3);
    const int n = p.L * p.B * p.H;  // below 2^31, checked at launch
    const uint32_t bar_state = smem_addr(smem + lay.bar()), bar_in = bar_state + 8;
    float *vec = reinterpret_cast<float *>(smem + lay.vec());
    float *sbeta = reinterpret_cast<float *>(smem + lay.beta());
    float *skq = reinterpret_cast<float *>(smem + lay.kq());

    if (tid == 0) {
        mbar_init(bar_state, 1);
        mbar_init(bar_in, NT + 1);
    }
    __syncthreads();
    int u = next_live(p, blockIdx.x, n);
    if (u < n) {
        if (tid == 0)
            prefetch_state(p, lay, smem, bar_state, u);
        prefetch_inputs(p, lay, smem, bar_in, u, tid);
    }
    uint32_t parity_state = 0, parity_in = 0;

    while (u < n) {
        const Unit x = unit_of(p, u);
        const int T = x.T;
        bool arrived = mbar_wait(bar_in, parity_in);
        if (__syncthreads_or(!arrived)) {
            if (tid == 0 && p.status)
                atomicOr(p.status, KDA_ST_TIMEOUT);
            mbar_wait(bar_in, parity_in);  // let copies in flight land before the CTA leaves
            mbar_wait(bar_state, parity_state);
            if (tid == 0)
                bulk_wait_all();
            return;
        }
        parity_in ^= 1u;

        // ---- prologue: conv + SiLU, norms, gates (one warp per row) ----------
        {
            const float4 *cw = reinterpret_cast<const float4 *>(smem + lay.stage_w());
            const int c0 = 4 * lane;
            // conv ring after the round (last 3 of [ring, rows]) and its snapshot; issued
            // first, they depend on nothing computed here
            float4 *rout = reinterpret_cast<float4 *>(p.ring_out + static_cast<size_t>(u) * 9 * D);
            float4 *rsnap = p.ring_snap ? reinterpret_cast<float4 *>(p.ring_snap + static_cast<size_t>(u) * 9 * D)
                                        : nullptr;
            for (int idx = tid; idx < 9 * D / 4; idx += NT) {
                const int s = idx / 96, slot = (idx % 96) / 32, c4 = idx % 32;
                rout[idx] = fetch4(lay, smem, s, T + slot, 4 * c4);
                if (rsnap)
                    rsnap[idx] = fetch4(lay, smem, s, slot, 4 * c4);
            }
            for (int t = wi; t < T; t += NW) {
                // the row's beta load goes out first; its latency hides behind the conv
                const float rb = lane == 0 ? load_scalar(p.xb, p.bf16, (static_cast<size_t>(x.lb) * p.T_rows + t) * p.H + x.h)
                                           : 0.f;
                float y[3][4];
#pragma unroll
                for (int s = 0; s < 3; ++s) {
                    const float4 x0 = fetch4(lay, smem, s, t, c0), x1 = fetch4(lay, smem, s, t + 1, c0);
                    const float4 x2 = fetch4(lay, smem, s, t + 2, c0), x3 = fetch4(lay, smem, s, t + 3, c0);
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
                const float4 rg = fetch4(lay, smem, 3, t + 3, c0);  // raw forget-gate row t
                const float rgv[4] = {rg.x, rg.y, rg.z, rg.w};
                float dv[4];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    dv[cc] = __expf(__fmul_rn(GATE_LOWER_BOUND, sigmoidf_(rgv[cc])));
                float *vt = vec + t * 4 * D + c0;
                *reinterpret_cast<float4 *>(vt) = make_float4(dv[0], dv[1], dv[2], dv[3]);
                *reinterpret_cast<float4 *>(vt + D) = make_float4(kh[0], kh[1], kh[2], kh[3]);
                *reinterpret_cast<float4 *>(vt + 2 * D) = make_float4(qh[0], qh[1], qh[2], qh[3]);
                *reinterpret_cast<float4 *>(vt + 3 * D) = make_float4(y[2][0], y[2][1], y[2][2], y[2][3]);
                if (lane == 0) {
                    skq[t] = kq;
                    sbeta[t] = sigmoidf_(rb);
                }
            }
        }
        // ---- state: stage -> registers ---------------------------------------------
        arrived = mbar_wait(bar_state, parity_state);
        if (__syncthreads_or(!arrived)) {
            if (tid == 0 && p.status)
                atomicOr(p.status, KDA_ST_TIMEOUT);
            mbar_wait(bar_state, parity_state);
            if (tid == 0)
                bulk_wait_all();
            return;
        }
        parity_state ^= 1u;
        if (tid == 0 && p.s_snap) {
            // the pre-round state leaves as a bulk store straight from the stage; the stage
            // holds only what the bulk load wrote, so no proxy fence is needed before it
            for (int c = 0; c < 4; ++c)
                bulk_store(p.s_snap + static_cast<size_t>(u) * D * D + c * 4096,
                           smem_addr(smem + lay.stage_state() + c * 16384), 16384);
            bulk_commit();
        }
        float2 S[8][4];  // S[rp][c] = (S[16rg + 2rp][jbase + c], S[16rg + 2rp + 1][jbase + c])
        {
            const float *Ss = reinterpret_cast<const float *>(smem + lay.stage_state());
#pragma unroll
            for (int rp = 0; rp < 8; ++rp) {
                const int i = 16 * rg + 2 * rp;
                const float4 a = *reinterpret_cast<const float4 *>(Ss + i * D + jbase);
                const float4 c = *reinterpret_cast<const float4 *>(Ss + (i + 1) * D + jbase);
                S[rp][0] = make_float2(a.x, c.x);
                S[rp][1] = make_float2(a.y, c.y);
                S[rp][2] = make_float2(a.z, c.z);
                S[rp][3] = make_float2(a.w, c.w);
            }
        }
        __syncthreads();  // every generic read of the stage is done; vec, beta, k.q are written

        // ---- refill the stage with the next unit while this one scans ----------------
        const int un = next_live(p, u + gridDim.x, n);
        // the next unit's state fetch waits until the snapshot store has read the stage
        bool state_due = un < n;
        if (state_due && !p.s_snap) {
            if (tid == 0) {
                fence_proxy_async();
                prefetch_state(p, lay, smem, bar_state, un);
            }
            state_due = false;
        }
        if (un < n)
            prefetch_inputs(p, lay, smem, bar_in, un, tid);

        // ---- the T-row gated delta rule -----------------------------------------
        float *outp = p.out ? p.out + (static_cast<size_t>(x.lb) * p.T_rows * p.H + x.h) * D + jsum : nullptr;
        const int b2 = rg >> 2, b1 = (rg >> 1) & 1, b0 = rg & 1;
        for (int t = 0; t < T; ++t) {
            const float *vt = vec + t * 4 * D;
            float2 uacc[4], eacc[4], kk[8];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                uacc[c] = eacc[c] = make_float2(0.f, 0.f);
            // S' = d S ;  u = S'^T k ;  e = S'^T q   (this thread's 16 rows)
#pragma unroll
            for (int rq = 0; rq < 4; ++rq) {
                const int ib = 16 * rg + 4 * rq;
                const float4 d4 = *reinterpret_cast<const float4 *>(vt + ib);
                const float4 k4 = *reinterpret_cast<const float4 *>(vt + D + ib);
                const float4 q4 = *reinterpret_cast<const float4 *>(vt + 2 * D + ib);
                const float2 dA = make_float2(d4.x, d4.y), dB = make_float2(d4.z, d4.w);
                const float2 qA = make_float2(q4.x, q4.y), qB = make_float2(q4.z, q4.w);
                kk[2 * rq] = make_float2(k4.x, k4.y);
                kk[2 * rq + 1] = make_float2(k4.z, k4.w);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    S[2 * rq][c] = __fmul2_rn(S[2 * rq][c], dA);
                    uacc[c] = __ffma2_rn(S[2 * rq][c], kk[2 * rq], uacc[c]);
                    eacc[c] = __ffma2_rn(S[2 * rq][c], qA, eacc[c]);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    S[2 * rq + 1][c] = __fmul2_rn(S[2 * rq + 1][c], dB);
                    uacc[c] = __ffma2_rn(S[2 * rq + 1][c], kk[2 * rq + 1], uacc[c]);
                    eacc[c] = __ffma2_rn(S[2 * rq + 1][c], qB, eacc[c]);
                }
            }
            // reduce-scatter over the 8 row groups: lane bit 4 splits u / e, bits 3 and 2
            // split the 4 columns; each sum ends on exactly one lane
            float v8[8];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                v8[c] = __fadd_rn(uacc[c].x, uacc[c].y);
                v8[4 + c] = __fadd_rn(eacc[c].x, eacc[c].y);
            }
            float v4[4], v2[2];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float keep = b2 ? v8[4 + m] : v8[m], send = b2 ? v8[m] : v8[4 + m];
                v4[m] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 16));
            }
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const float keep = b1 ? v4[2 + m] : v4[m], send = b1 ? v4[m] : v4[2 + m];
                v2[m] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 8));
            }
            const float keep1 = b0 ? v2[1] : v2[0], send1 = b0 ? v2[0] : v2[1];
            const float sum = __fadd_rn(keep1, __shfl_xor_sync(0xffffffffu, send1, 4));
            // u lanes: w = beta (v - u); e lanes: o = (e + w (k.q)) / sqrt(128)
            const float w = __fmul_rn(sbeta[t], __fsub_rn(vt[3 * D + jsum], sum));
            const float w_of_col = __shfl_xor_sync(0xffffffffu, w, 16);
            if (outp && b2)
                outp[static_cast<size_t>(t) * p.H * D] = __fmul_rn(__fmaf_rn(w_of_col, skq[t], sum), OUT_SCALE);
            // every lane gathers w of its 4 columns from the u lanes 4c + cg
            float2 wc[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float wv = __shfl_sync(0xffffffffu, w, 4 * c + cg);
                wc[c] = make_float2(wv, wv);
            }
            // S = S' + k w^T
#pragma unroll
            for (int rp = 0; rp < 8; ++rp)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    S[rp][c] = __ffma2_rn(kk[rp], wc[c], S[rp][c]);
            if (state_due && t == (T > 1 ? 1 : 0)) {
                if (tid == 0) {
                    bulk_wait_read();  // the snapshot store is done with the stage
                    fence_proxy_async();
                    prefetch_state(p, lay, smem, bar_state, un);
                }
                state_due = false;
            }
        }

        // ---- state write-back ---------------------------------------------------
        {
            float *So = p.s_out + static_cast<size_t>(u) * D * D;
#pragma unroll
            for (int rp = 0; rp < 8; ++rp) {
                const int i = 16 * rg + 2 * rp;
                *reinterpret_cast<float4 *>(So + i * D + jbase) =
                    make_float4(S[rp][0].x, S[rp][1].x, S[rp][2].x, S[rp][3].x);
                *reinterpret_cast<float4 *>(So + (i + 1) * D + jbase) =
                    make_float4(S[rp][0].y, S[rp][1].y, S[rp][2].y, S[rp][3].y);
            }
        }
        __syncthreads();  // vec, beta, k.q are free for the next unit's prologue
        u = un;
    }
    if (tid == 0)
        bulk_wait_all();  // the last snapshot stores leave before the CTA's shared memory does
}

struct DeviceInfo {
    int sms = 0;
    int smem_set = 0;
    int per_sm[2][KDA_TMAX + 1] = {};  // CTAs per SM by (raw element size 2/4, rows)
};

int launch_scan(const ScanParams &p, int tcap, cudaStream_t stream)
{
    const long long units = static_cast<long long>(p.L) * p.B * p.H;
    if (units == 0)
        return ok();
    if (units > 0x7fffffffLL - 4LL * 152 * 64)
        return fail(KDA_EINVAL, "L*B*H exceeds the unit index range");
    const Layout lay{tcap, p.bf16 ? 2 : 4};
    const size_t smem = lay.total();
    static DeviceInfo info[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(KDA_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64)
        return fail(KDA_EINVAL, "device ordinal beyond the launch table");
    DeviceInfo &di = info[dev];
    if (di.sms == 0) {
        e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return fail(KDA_ECUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
    }
    if (di.smem_set < static_cast<int>(smem)) {
        const size_t most = Layout{KDA_TMAX, 4}.total();
        e = cudaFuncSetAttribute(kda_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(most));
        if (e != cudaSuccess)
            return fail(KDA_ECUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
        di.smem_set = static_cast<int>(most);
    }
    int &per_sm = di.per_sm[p.bf16 ? 0 : 1][tcap];
    if (per_sm == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_scan_kernel, NT, smem);
        if (e != cudaSuccess || per_sm < 1) {
            per_sm = 0;
            return fail(KDA_ECUDA, "kda_scan_kernel does not fit on an SM");
        }
    }
    const long long grid = std::min<long long>(units, static_cast<long long>(di.sms) * per_sm);
    kda_scan_kernel<<<static_cast<unsigned>(grid), NT, smem, stream>>>(p);
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
