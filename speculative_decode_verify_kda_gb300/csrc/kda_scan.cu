// kda_scan.cu -- the fused KDA verify walk (short conv, activations, gated delta
// rule) for sm_103a, and the accept-j rollback that replays it.
//
// A unit is one (layer, session, head): its 128 x 128 f32 state, the raw rows of
// its T drafted positions, its conv ring and conv weights.  One persistent CTA per
// SM walks the units blockIdx.x, +gridDim.x, ... with two kinds of warps that hand
// work to each other through mbarriers in shared memory:
//
//   prologue warps (4) one per stream (q, k, v, g), one unit ahead of the scan:
//                      width-4 causal conv + SiLU of q, k, v (mini fixture
//                      linear_attn_config of glm5_spec_ppn_gate.rs:
//                      short_conv_kernel_size 4, head_dim 128, gate_lower_bound
//                      -5.0) sliding along the rows in registers, the L2 norms of
//                      q and k, the forget gate d = exp(-5 sigmoid(raw_g))
//                      and beta = sigmoid(raw_beta), written as the round's scan
//                      inputs into one of two shared buffers; they also re-roll
//                      the conv ring (and snapshot it).  The g warp also stages the
//                      raw q, k, v, g rows with 1D bulk copies, one or two units
//                      ahead, once the prologue is done with a stage.
//   scan warps (8)     hold the unit's state in registers for its whole T-row
//                      loop and write it back once: each 64 KiB head state
//                      crosses HBM once in and once out per round (plus the
//                      snapshot copy of the in-place verify).  Output rows go
//                      straight to global memory.  Scan warp 0 also loads the
//                      states: a unit's state arrives as four 2D tensor copies (32
//                      columns x 128 rows each, 128-byte swizzle) into one of two
//                      slots, two units ahead, and leaves again from the slot as
//                      four tensor stores to the snapshot (the fused snapshot write).
// Twelve warps put three on each SM sub-partition, which leaves 168 registers per
// thread for the scan warps' 64-element tiles (thirteen would cap them at 128).
//
// Register tile: lane 4 rg + cg of scan warp wi holds key rows rg + 8 r (r < 16)
// of value columns 16 wi + 4 cg .. +3, column pairs packed into float2 so each
// element operation is one lane of a packed f32x2 instruction (__fmul2_rn,
// __ffma2_rn) and each row of the tile is the 16-byte vector it is loaded from and
// stored as (a row-pair packing needs register moves against those vectors, which
// cost the T-loop 40 %).  The row scalars d, k, q are broadcast into both halves of
// a pair.  Rows rg + 8 r share their 128-byte swizzle phase.  The scan inputs of a
// row hold each row group's d, k and q contiguously, so a quarter warp reads two
// broadcast addresses per load.
// Per row t (glm_spec.rs module doc, VERIFY-ROW BATCHING: the recurrence stays
// sequential inside one launch, the in-kernel T-loop being the chained t=1
// program):
//   S' = d_t (.) S               d = exp(g)
//   u  = S'^T k,  e = S'^T q     one register sweep (which also sums k.q), then a
//                                3-step shuffle reduce-scatter over the 8 row groups
//   w  = beta (v - u)
//   o  = (e + w (k.q)) / sqrt(128)   == (S' + k w^T)^T q / sqrt(128)
//   S  = S' + k w^T              second register sweep
// Every operation is an explicitly rounded intrinsic and the code for a row does
// not depend on T, on the unit or on whether outputs are written, so T rows in one
// launch and T launches of one row give the same bits, and so do a rollback
// replay and a fresh verify.
//
// Rollback runs the same kernel from the snapshot over rows 0..keep-1 of the
// stashed raw rows (the conv re-runs inside the replay), with outputs and the
// snapshot store switched off.  A deferred round runs that replay and the next
// round's rows as two items of one unit, the state staying in registers between
// them.  Rounds whose length differs per session run each unit's own row count in
// the same grid.  A second instantiation also writes the column stash (the state
// and ring after every row).
// Every wait on an mbarrier is bounded by one second.  A wait that runs out sets
// KDA_ST_TIMEOUT (where the call has a status word) and a shared abort flag that
// ends every warp of the CTA; the warps that issue copies first let theirs land.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>
#include <unordered_map>
#include <cstring>
#include <string>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int D = 128;
constexpr int NSCAN = 8;                   // scan warps; warp 0 also loads the states
constexpr int NPRO = 4;                    // prologue warps: q, k, v, g; g also stages the raw rows
constexpr int NT = (NSCAN + NPRO) * 32;    // 12 warps: 3 per SM sub-partition, so up to 168 registers
constexpr int GRP = 52;                    // floats per row group of a scan-input row: d, k, q (16 each), pad
constexpr int SI_V = 8 * GRP;              // offset of v (natural order) in a scan-input row
constexpr int SI_ROW = SI_V + D;           // floats per scan-input row
constexpr float L2_EPS = 1e-6f;
constexpr float GATE_LOWER_BOUND = -5.0f;
constexpr float OUT_SCALE = 0.0883883476483184405501f;  // 1 / sqrt(128)
constexpr uint64_t WAIT_NS = 1000000000ull;  // an mbarrier wait gives up after one second

// mbarriers: state slots full/empty, scan-input buffers full/empty, and raw-row stage
// b of stream s full (B_STG_FULL + 4 b + s: each prologue warp stages its own stream)
enum { B_STATE_FULL = 0, B_STATE_EMPTY = 2, B_SI_FULL = 4, B_SI_EMPTY = 6, B_STG_FULL = 8, NBARS = 16 };

// Rows a unit runs: KEEP_NONE all T_run; ROWS_* a verify with per-session row counts
// (host values in keep_host, or rows_dev); KEEP_* a rollback to per-session keep;
// DEFERRED a verify of T_run rows that first replays the previous round's kept rows
// (keep_dev holds the previous round's keep, T_prev its row count).
enum KeepMode { KEEP_NONE = 0, KEEP_HOST = 1, KEEP_DEVICE = 2, ROWS_HOST = 3, ROWS_DEVICE = 4, DEFERRED = 5 };

// Division by a fixed divisor d as a multiply and shift (Granlund and Montgomery,
// "Division by invariant integers using multiplication", 1994, round-up method):
// with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1, n / d = (mulhi(n, m) + n)
// >> l for every 32-bit n.  The unit index walks divide by H and B several times per
// work item, and a general integer division is a long instruction sequence.
struct FastDiv {
    uint32_t d, m, l;
};

struct ScanParams {
    CUtensorMap tm_in;     // state read: [units * 128 rows][128] f32, box 32 x 128, 128B swizzle
    CUtensorMap tm_in2;    // DEFERRED: the state read of units with nothing to replay
    CUtensorMap tm_snap;   // snapshot write, same geometry (unused without s_snap)
    CUtensorMap tm_rows[4];  // raw rows q, k, v, g: [L*B][T_rows][H][128], box 128 x 1 x T_rows x 1
    CUtensorMap tm_prev[4];  // DEFERRED: the previous round's raw rows, box 128 x 1 x T_prev x 1
    CUtensorMap tm_copy[4];  // rows_host: the device copy of this call's raw rows, as tm_rows
    float *s_out;          // [L][B][H][D][D]
    float *s_snap;         // nullable: receives the state read through tm_in
    const float *ring_in;  // [L][B][H][3][3][D]
    float *ring_out;
    float *ring_snap;      // nullable: receives ring_in of each unit
    const float *conv_w;   // [L][H][3][D][4]
    const void *xq, *xk, *xv, *xg, *xb;  // [L][B][T_rows][H][D], xb [L][B][T_rows][H]
    float *out;            // nullable: [L][B][T_rows][H][D]
    float *s_snap_out;     // DEFERRED: receives the state after the replay (this round's snapshot)
    const float *ring_in2; // DEFERRED: the ring of units with nothing to replay
    float *ring_snap_out;  // DEFERRED: receives the ring after the replay
    const void *xb_prev;   // DEFERRED: the previous round's raw beta [L][B][T_prev][H]
    void *copy_beta;       // rows_host: the device copy of this call's raw beta
    float *w_out;          // nullable: [L][B][T_rows][H][D], the update vector w_t of every verify row
    const float *w_in;     // nullable: the update vectors of the rows a replay re-runs, [L][B][T_w][H][D]
    int T_w;               // row count of w_in (the replayed round's T)
    float *s_cols;         // nullable: [L][B][H][T_rows][D][D], the state after each row
    float *ring_cols;      // with s_cols: [L][B][H][T_rows][3][3][D], the ring after each row
    const int *keep_dev;   // KEEP_DEVICE: [B]
    const int *rows_dev;   // ROWS_DEVICE, or KEEP_DEVICE after a per-session round: [B] row counts
    int *status;           // nullable device status word
    const unsigned *ready; // nullable: this call's raw rows of (layer, session) pair lb = l B + b
                           // are in place once ready[lb / ready_ppf] has reached epoch
    unsigned epoch;
    int ready_ppf;
    int L, B, H;
    FastDiv divH, divB;    // u / H and lb / B
    int T_rows;            // row count of the raw-row tensors
    int T_run;             // rows to run for KEEP_NONE and DEFERRED
    int T_prev;            // DEFERRED: row count of the previous round's raw-row tensors
    int tcap;              // most rows any unit runs (sizes the buffers)
    int nstg;              // raw-row stages: 2 where shared memory allows, else 1
    int bf16;
    int rows_host;         // this call's raw rows (xq..xb) are read in place from host memory
    int keep_mode;
    unsigned char keep_host[KDA_HOST_KEEP_MAX];
};

// Shared memory, from a 1024-byte aligned base (the 128-byte swizzle repeats
// every 1024 bytes): two 64 KiB state slots, two scan-input buffers of tcap rows,
// their beta scalars, nstg raw-row stages [4 streams][tcap][128], the
// mbarriers and the abort flag.
struct Layout {
    int tcap, es, nstg;
    __host__ __device__ size_t slot(int s) const { return static_cast<size_t>(s) * D * D * 4; }
    __host__ __device__ size_t si(int b) const { return slot(2) + static_cast<size_t>(b) * tcap * SI_ROW * 4; }
    __host__ __device__ size_t sc(int b) const { return si(2) + static_cast<size_t>(b) * 16 * 8; }
    __host__ __device__ size_t row_bytes() const { return static_cast<size_t>(D) * es; }
    __host__ __device__ size_t stg(int b) const { return sc(2) + static_cast<size_t>(b) * 4 * tcap * row_bytes(); }
    __host__ __device__ size_t bars() const { return stg(nstg); }
    __host__ __device__ size_t flag() const { return bars() + NBARS * 8; }
    __host__ __device__ size_t total() const { return flag() + 16 + 1024; }  // + alignment slack
};

// sigmoid through the fast exp2 / reciprocal intrinsics: relative error ~1e-6, far
// inside the 1e-4 parity bar, and a short dependency chain
__device__ __forceinline__ float sigmoidf_(float z)
{
    return __fdividef(1.0f, __fadd_rn(1.0f, __expf(-z)));
}

__device__ __forceinline__ float silu(float a) { return __fmul_rn(a, sigmoidf_(a)); }

__device__ __forceinline__ float load_scalar(const void *base, int bf16, size_t idx)
{
    if (bf16)
        return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t *>(base)[idx]) << 16);
    return static_cast<const float *>(base)[idx];
}

__device__ __forceinline__ float conv4(float4 w, float x0, float x1, float x2, float x3)
{
    // w.x multiplies x[t-3] (x0), w.w the current row x[t] (x3)
    return __fmaf_rn(w.w, x3, __fmaf_rn(w.z, x2, __fmaf_rn(w.y, x1, __fmul_rn(w.x, x0))));
}

// ---- TMA, bulk copies and mbarriers ------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// 2D tensor copy global -> shared of the box at (x, y), counted in bytes by `bar`
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, int x, int y, uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar) : "memory");
}

// 4D tensor copy global -> shared of the box at (c0, c1, c2, c3), counted in bytes by `bar`
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *tm, int c0, int c1, int c2, int c3,
                                            uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4, %5}], [%6];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
                 : "memory");
}

// L2 prefetch of the 2D / 4D box at the given coordinates (a hint: no data is consumed,
// so it may run before the previous kernel's results are visible)
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *tm, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 ::"l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y) : "memory");
}

__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap *tm, int c0, int c1, int c2, int c3)
{
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];"
                 ::"l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3) : "memory");
}

// 4D tensor copy shared -> global of the box at (c0, c1, c2, c3), tracked by bulk groups
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *tm, int c0, int c1, int c2, int c3, uint32_t src)
{
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];"
                 ::"l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src) : "memory");
}

// 2D tensor copy shared -> global of the box at (x, y), tracked by bulk groups
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *tm, int x, int y, uint32_t src)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(src) : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// the bulk stores issued so far have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// the bulk stores issued so far are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared control block of a CTA: mbarrier base address, abort flag, status word.
struct Ctl {
    uint32_t bars;
    volatile int *abort;
    int *status;
    __device__ uint32_t bar(int i) const { return bars + 8u * i; }
};

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded warp-wide wait for the phase of barrier `i` with `parity`.  Every lane
// acquires the phase itself; the warp leaves together.  False once the CTA is
// aborting, or after WAIT_NS of waiting (which starts the abort).
__device__ bool warp_wait(const Ctl &c, int i, uint32_t parity)
{
    const uint32_t a = c.bar(i);
    if (__all_sync(0xffffffffu, mbar_try(a, parity)))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (__all_sync(0xffffffffu, mbar_try(a, parity)))
            return true;
        if ((n & 15) == 0) {
            if (__any_sync(0xffffffffu, *c.abort != 0))
                return false;
            if (__any_sync(0xffffffffu, globaltimer_ns() - t0 > WAIT_NS))
                break;
        }
        if (n >= 64)
            __nanosleep(128);
    }
    if ((threadIdx.x & 31) == 0) {
        if (c.status)
            atomicOr(c.status, KDA_ST_TIMEOUT);
        *c.abort = 1;
    }
    return false;
}

// The same bounded wait for one thread that must not leave early (copies in flight).
__device__ bool drain_wait(uint32_t a, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 0;; ++n) {
        if (mbar_try(a, parity))
            return true;
        if ((n & 15) == 0 && globaltimer_ns() - t0 > WAIT_NS)
            return false;
        if (n >= 64)
            __nanosleep(128);
    }
}

// ---- units --------------------------------------------------------------------------
struct Unit {
    int h, b, l, T;
    int R;         // DEFERRED: the previous round's rows to replay first (0: none)
    long long lb;  // l * B + b
};

// rows unit u runs: > 0 to run, 0 nothing to do, -1 an invalid device keep or row
// count.  The plain verify comes first: this runs for every unit in every warp.
__device__ __forceinline__ int unit_rows(const ScanParams &p, int b)
{
    if (p.keep_mode == KEEP_NONE)
        return p.T_run;
    if (p.keep_mode == KEEP_HOST) {
        const int kp = p.keep_host[b];  // validated on the host; T_rows where nothing is to do
        return kp >= p.T_rows ? 0 : kp;
    }
    if (p.keep_mode == KEEP_DEVICE) {
        const int kp = p.keep_dev[b];
        const int tb = p.rows_dev ? p.rows_dev[b] : p.T_rows;  // the session's rows in the round
        if (tb < 1 || tb > p.T_rows || kp < 1 || kp > tb)
            return -1;
        return kp == tb ? 0 : kp;
    }
    if (p.keep_mode == ROWS_HOST)
        return p.keep_host[b];  // validated 1..T_rows on the host
    if (p.keep_mode == DEFERRED) {
        const int kp = p.keep_dev[b];
        return kp < 1 || kp > p.T_prev ? -1 : p.T_run;
    }
    const int tb = p.rows_dev[b];  // ROWS_DEVICE
    return tb < 1 || tb > p.T_rows ? -1 : tb;
}

// Whether item `part` of a unit re-runs rows of an earlier verify (the replay of a
// rollback, or a deferred round's first item), whose update vectors w_in may hold.
__device__ __forceinline__ bool is_replay(const ScanParams &p, int part)
{
    return part == 0 || p.keep_mode == KEEP_HOST || p.keep_mode == KEEP_DEVICE;
}

// DEFERRED: the previous round's rows session b replays before its verify (0 when it
// kept them all); 0 in every other mode.
__device__ __forceinline__ int replay_rows(const ScanParams &p, int b)
{
    if (p.keep_mode != DEFERRED)
        return 0;
    const int kp = p.keep_dev[b];
    return kp < p.T_prev ? kp : 0;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, FastDiv f)
{
    return static_cast<uint32_t>((static_cast<uint64_t>(__umulhi(n, f.m)) + n) >> f.l);
}

// the session of unit u = (l * B + b) * H + h
__device__ __forceinline__ int session_of(const ScanParams &p, int u)
{
    const uint32_t lb = fdiv(static_cast<uint32_t>(u), p.divH);
    return static_cast<int>(lb - fdiv(lb, p.divB) * static_cast<uint32_t>(p.B));
}

__device__ __forceinline__ Unit unit_of(const ScanParams &p, int u)
{
    Unit x;
    const uint32_t lb = fdiv(static_cast<uint32_t>(u), p.divH);
    const uint32_t l = fdiv(lb, p.divB);
    x.h = static_cast<int>(static_cast<uint32_t>(u) - lb * static_cast<uint32_t>(p.H));
    x.lb = lb;
    x.b = static_cast<int>(lb - l * static_cast<uint32_t>(p.B));
    x.l = static_cast<int>(l);
    x.T = unit_rows(p, x.b);
    x.R = replay_rows(p, x.b);
    return x;
}

// A unit's work items: part 0 the replay of the previous round's kept rows (DEFERRED
// units with rows to replay), part 1 this call's rows.  Items pass through the
// raw-row stages and scan-input buffers in order; a unit's state stays in the scan
// warps' registers from its first item to its last.
struct Item {
    int u, part;
};

__device__ __forceinline__ Item first_item(const ScanParams &p, int u, int n)
{
    return Item{u, u < n && replay_rows(p, session_of(p, u)) > 0 ? 0 : 1};
}

// The first unit at or after u (stepping by the grid) that has rows to run.  Every
// warp walks the same sequence; only lane 0 of scan warp 0 reports bad keeps.
__device__ int next_live(const ScanParams &p, int u, int n, bool report)
{
    for (; u < n; u += gridDim.x) {
        const int T = unit_rows(p, session_of(p, u));
        if (T > 0)
            return u;
        if (T < 0 && report && p.status)
            atomicOr(p.status, KDA_ST_BADKEEP);  // the session is left untouched
    }
    return n;
}

__device__ __forceinline__ Item next_item(const ScanParams &p, Item it, int n)
{
    if (it.part == 0)
        return Item{it.u, 1};
    return first_item(p, next_live(p, it.u + gridDim.x, n, false), n);
}

// Staged raw rows: before a prologue warp copies an item's rows of this call (part 1)
// it waits, bounded like warp_wait, until the flag of the item's range of (layer,
// session) pairs has reached the call's epoch.  The flag is written by a stream memory operation after the rows'
// host-to-device copy on another stream (no kernel writes it).  Lane 0 reads it with
// acquire semantics; the proxy fence orders the tensor copies that follow after it.  A
// warp walks its units in increasing (layer, session) order, so it reads each flag
// once: last_f is the flag it saw set last.
__device__ bool rows_ready(const ScanParams &p, const Ctl &c, int u, int part, int lane, int &last_f)
{
    if (!p.ready || part == 0)
        return true;
    const int fi = static_cast<int>(fdiv(static_cast<uint32_t>(u), p.divH)) / p.ready_ppf;
    if (fi == last_f)
        return true;
    int ok = 1;
    if (lane == 0) {
        const unsigned *f = p.ready + fi;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t n = 0;; ++n) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
            if (static_cast<int>(v - p.epoch) >= 0)
                break;
            if ((n & 15) == 15) {
                if (*c.abort != 0) {
                    ok = 0;
                    break;
                }
                if (globaltimer_ns() - t0 > WAIT_NS) {
                    if (c.status)
                        atomicOr(c.status, KDA_ST_TIMEOUT);
                    *c.abort = 1;
                    ok = 0;
                    break;
                }
            }
            __nanosleep(n < 64 ? 32 : 256);
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    if (ok)
        last_f = fi;
    return ok != 0;
}

// ---- copies issued by scan warp 0 (states) and the prologue warps (raw rows) ----------
// Unit u's 64 KiB state into a slot: four boxes of 32 columns x 128 rows (lane 0).  A
// DEFERRED unit with nothing to replay starts from the other buffer (tm_in2).
__device__ __forceinline__ void issue_state(const ScanParams &p, uint32_t slot, uint32_t bar, int u)
{
    const CUtensorMap *tm =
        p.keep_mode == DEFERRED && replay_rows(p, session_of(p, u)) == 0 ? &p.tm_in2 : &p.tm_in;
    mbar_expect_tx(bar, D * D * 4);
#pragma unroll
    for (int b = 0; b < 4; ++b)
        tma_load_2d(slot + b * 16384, tm, 32 * b, u * D, bar);
}

// An item's raw rows of stream s (0 q, 1 k, 2 v, 3 g) into the stage: one tensor copy
// of all rows of its head in the round it belongs to (a unit that runs fewer rows
// gets them all; the rest are not read).  Lane 0 arms the barrier with the byte
// count; each prologue warp stages its own stream, with a barrier per stream and stage.
template <bool HR>
__device__ void issue_stream(const ScanParams &p, const Layout &lay, uint32_t stg, uint32_t bar, Item it, int s,
                             int lane)
{
    const int lb = static_cast<int>(fdiv(static_cast<uint32_t>(it.u), p.divH)), h = it.u - lb * p.H;
    const uint32_t rb = static_cast<uint32_t>(lay.row_bytes());
    if (HR && it.part == 1) {
        // rows in host memory: asynchronous 16-byte copies per lane that the barrier
        // tracks (the SM reads host memory like global memory), once the device copy of
        // the stage's previous item has read the stage
        if (lane == 0)
            bulk_wait_read();
        __syncwarp();
        // 16 bytes a lane: a bf16 row (256 bytes) is half a warp, so a warp copies two rows
        // an instruction
        const int lpr = static_cast<int>(rb / 16);  // lanes a row: 16 (bf16) or 32 (f32)
        const int sub = lane % lpr, r0 = lane / lpr, rstep = 32 / lpr;
        const char *base = static_cast<const char *>(s == 0 ? p.xq : s == 1 ? p.xk : s == 2 ? p.xv : p.xg);
        const char *src = base + (static_cast<size_t>(lb) * p.T_rows * p.H + h) * rb + sub * 16;
        const size_t pitch = static_cast<size_t>(p.H) * rb;
        const uint32_t dst = stg + s * lay.tcap * rb + sub * 16;
        for (int t = r0; t < p.T_rows; t += rstep)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + t * rb), "l"(src + t * pitch)
                         : "memory");
        asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar);  // the barrier's one arrival; it completes once the copies land
        return;
    }
    fence_proxy_async();  // the prologue's generic reads of the stage come first
    if (lane == 0) {
        if (HR)
            bulk_wait_read();  // and the device copy of the stage's previous item has read it
        mbar_expect_tx(bar, static_cast<uint32_t>(it.part == 0 ? p.T_prev : p.T_rows) * rb);
        tma_load_4d(stg + s * lay.tcap * rb, it.part == 0 ? &p.tm_prev[s] : &p.tm_rows[s], 0, h, 0, lb, bar);
    }
}

// rows_host: the device copy of an item's rows of stream s, sent from the stage once
// they have landed (the stash records the copy for the next round's replay).
__device__ __forceinline__ void copy_stage_out(const ScanParams &p, const Layout &lay, uint32_t stg, int u, int s,
                                               int lane)
{
    const int lb = static_cast<int>(fdiv(static_cast<uint32_t>(u), p.divH)), h = u - lb * p.H;
    fence_proxy_async();  // the stage's rows, landed, before the tensor store reads them
    __syncwarp();
    if (lane == 0) {
        tma_store_4d(&p.tm_copy[s], 0, h, 0, lb, stg + s * lay.tcap * static_cast<uint32_t>(lay.row_bytes()));
        bulk_commit();
    }
}

// ---- prologue warps -----------------------------------------------------------------
// What a prologue lane loads for an item before it needs it: for q, k, v the conv
// weights of its 4 channels and, for a unit's first item, their ring slots; for g the
// raw beta of row `lane` of the item's round.
struct Pre {
    float4 w[4];     // w[m]: the 4 taps of channel 4 lane + m
    float4 ring[3];  // ring slot 0 (oldest) .. 2 of channels 4 lane .. +3
    float beta;
};

template <bool HR>
__device__ __forceinline__ void load_pre(const ScanParams &p, Item it, int pw, int lane, Pre &pr)
{
    const Unit x = unit_of(p, it.u);
    if (pw < 3) {
        const float4 *w = reinterpret_cast<const float4 *>(p.conv_w) +
                          ((static_cast<size_t>(x.l) * p.H + x.h) * 3 + pw) * D + 4 * lane;
#pragma unroll
        for (int m = 0; m < 4; ++m)
            pr.w[m] = w[m];
        if (it.part == 0 || x.R == 0) {  // a verify item after a replay continues its window
            const float *src = p.keep_mode == DEFERRED && it.part == 1 ? p.ring_in2 : p.ring_in;
            const float4 *r = reinterpret_cast<const float4 *>(src + (static_cast<size_t>(it.u) * 3 + pw) * 3 * D) + lane;
#pragma unroll
            for (int sl = 0; sl < 3; ++sl)
                pr.ring[sl] = r[sl * (D / 4)];
        }
    } else {
        const int T = it.part == 0 ? x.R : x.T, trows = it.part == 0 ? p.T_prev : p.T_rows;
        const void *xb = it.part == 0 ? p.xb_prev : p.xb;
        const size_t bi = (static_cast<size_t>(x.lb) * trows + lane) * p.H + x.h;
        // host rows: every row's beta, for the device copy the prologue writes once it
        // has used the value (a store right here would wait for the host read)
        pr.beta = lane < (HR && it.part == 1 ? p.T_rows : T) ? load_scalar(xb, p.bf16, bi) : 0.f;
    }
}

// channels 4 lane .. +3 of raw row t of stream s in the stage, widened to f32
__device__ __forceinline__ float4 stage4(const unsigned char *stg, const Layout &lay, int s, int t, int lane)
{
    const unsigned char *r = stg + (static_cast<size_t>(s) * lay.tcap + t) * lay.row_bytes();
    if (lay.es == 4)
        return reinterpret_cast<const float4 *>(r)[lane];
    const uint2 v = reinterpret_cast<const uint2 *>(r)[lane];
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                       __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
}

// Key channel i of a d / k-hat / q-hat vector sits at row group i % 8, slot i / 8
// of a scan-input row (blocks at 0, 16, 32 of the group), so a scan thread finds
// its 16 rows i = rg + 8 r contiguous.  Lane's channels 4 lane + m have
// i % 8 = 4 (lane & 1) + m and i / 8 = lane / 2.
__device__ __forceinline__ void store_perm(float *row, int block, int lane, float4 v)
{
    float *g = row + 4 * (lane & 1) * GRP + block + (lane >> 1);
    g[0] = v.x;
    g[GRP] = v.y;
    g[2 * GRP] = v.z;
    g[3 * GRP] = v.w;
}

// The conv window of stream pw after an item's T rows without the conv itself (the
// last 3 raw inputs of [window, rows]): writes the ring after the item to ring_dst and,
// when snapshotting, the ring before it.
__device__ void roll_window(const ScanParams &p, const Layout &lay, const unsigned char *stg, float4 (&win)[3], int u,
                            int T, int pw, int lane, float *ring_dst)
{
    const size_t rbase = (static_cast<size_t>(u) * 3 + pw) * 3 * D;
    if (p.ring_snap) {
        float4 *rs = reinterpret_cast<float4 *>(p.ring_snap + rbase) + lane;
        rs[0] = win[0];
        rs[D / 4] = win[1];
        rs[2 * D / 4] = win[2];
    }
    const float4 r0 = T >= 3 ? stage4(stg, lay, pw, T - 3, lane) : T == 2 ? win[2] : win[1];
    const float4 r1 = T >= 2 ? stage4(stg, lay, pw, T - 2, lane) : win[2];
    const float4 r2 = stage4(stg, lay, pw, T - 1, lane);
    float4 *ro = reinterpret_cast<float4 *>(ring_dst + rbase) + lane;
    ro[0] = r0;
    ro[D / 4] = r1;
    ro[2 * D / 4] = r2;
    win[0] = r0;
    win[1] = r1;
    win[2] = r2;
}

// Stream pw (0 q, 1 k, 2 v) of one item: the conv window slides along the rows in
// registers, four rows at a time with no branch around the arithmetic (rows past T
// repeat row T-1 and are not stored), so the four rows' dependency chains overlap.
// win holds the window (the last 3 raw inputs) before the item and after it.  Writes
// the scan inputs (q-hat, k-hat or v), the ring after the item to ring_dst and, when
// snapshotting, the ring before it.
template <bool COLS>
__device__ void conv_stream(const ScanParams &p, const Layout &lay, const unsigned char *stg, float *si,
                            const float4 (&wt)[4], float4 (&win)[3], int u, int T, int pw, int lane, float *ring_dst)
{
    const size_t rbase = (static_cast<size_t>(u) * 3 + pw) * 3 * D;
    if (p.ring_snap) {
        float4 *rs = reinterpret_cast<float4 *>(p.ring_snap + rbase) + lane;
        rs[0] = win[0];
        rs[D / 4] = win[1];
        rs[2 * D / 4] = win[2];
    }
    // the window before row t0: x[t0-3], x[t0-2], x[t0-1] of the sequence [ring, rows]
    float4 x0 = win[0], x1 = win[1], x2 = win[2];
    const int block = pw == 0 ? 32 : 16;
    for (int t0 = 0; t0 < T; t0 += 4) {
        float4 W[7];  // the sequence from x[t0-3]: W[j .. j+3] is row t0+j's window
        W[0] = x0;
        W[1] = x1;
        W[2] = x2;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            W[3 + j] = stage4(stg, lay, pw, min(t0 + j, T - 1), lane);
        float4 y[4];
        float ss[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // w.x multiplies x[t-3], w.w the current row
            y[j].x = silu(conv4(wt[0], W[j].x, W[j + 1].x, W[j + 2].x, W[j + 3].x));
            y[j].y = silu(conv4(wt[1], W[j].y, W[j + 1].y, W[j + 2].y, W[j + 3].y));
            y[j].z = silu(conv4(wt[2], W[j].z, W[j + 1].z, W[j + 2].z, W[j + 3].z));
            y[j].w = silu(conv4(wt[3], W[j].w, W[j + 1].w, W[j + 2].w, W[j + 3].w));
            ss[j] = __fmaf_rn(y[j].w, y[j].w, __fmaf_rn(y[j].z, y[j].z, __fmaf_rn(y[j].y, y[j].y, __fmul_rn(y[j].x, y[j].x))));
        }
        if (COLS) {  // the ring after row t0 + j: W[j+1 .. j+3]
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (t0 + j < T) {
                    float4 *rc = reinterpret_cast<float4 *>(
                                     p.ring_cols + ((static_cast<size_t>(u) * p.T_rows + t0 + j) * 3 + pw) * 3 * D) +
                                 lane;
                    rc[0] = W[j + 1];
                    rc[D / 4] = W[j + 2];
                    rc[2 * D / 4] = W[j + 3];
                }
        }
        if (pw == 2) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (t0 + j < T)
                    *reinterpret_cast<float4 *>(si + (t0 + j) * SI_ROW + SI_V + 4 * lane) = y[j];
        } else {
            // the four rows' sums of squares reduce together (one fixed butterfly per row)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    ss[j] = __fadd_rn(ss[j], __shfl_xor_sync(0xffffffffu, ss[j], off));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float r = rsqrtf(__fadd_rn(ss[j], L2_EPS));
                const float4 yn = make_float4(__fmul_rn(y[j].x, r), __fmul_rn(y[j].y, r), __fmul_rn(y[j].z, r),
                                              __fmul_rn(y[j].w, r));
                if (t0 + j < T)
                    store_perm(si + (t0 + j) * SI_ROW, block, lane, yn);
            }
        }
        x0 = W[4];
        x1 = W[5];
        x2 = W[6];
    }
    // the ring after the item: x[T-3], x[T-2], x[T-1] of the sequence [window, rows]
    const float4 r0 = T >= 3 ? stage4(stg, lay, pw, T - 3, lane) : T == 2 ? win[2] : win[1];
    const float4 r1 = T >= 2 ? stage4(stg, lay, pw, T - 2, lane) : win[2];
    const float4 r2 = stage4(stg, lay, pw, T - 1, lane);
    float4 *ro = reinterpret_cast<float4 *>(ring_dst + rbase) + lane;
    ro[0] = r0;
    ro[D / 4] = r1;
    ro[2 * D / 4] = r2;
    win[0] = r0;
    win[1] = r1;
    win[2] = r2;
}

// A replayed item whose verify stored its update vectors: the v warp copies w_t of
// every row into the v slot of the scan-input row (natural order), which the replay
// loop reads instead of forming u and w again.  Four rows' loads in flight at a time
// (loading every row one item ahead held 60 more registers and measured slower).
__device__ void copy_w_rows(const ScanParams &p, float *si, int u, int T, int lane)
{
    const int lb = static_cast<int>(fdiv(static_cast<uint32_t>(u), p.divH)), h = u - lb * p.H;
    const float4 *src = reinterpret_cast<const float4 *>(p.w_in + (static_cast<size_t>(lb) * p.T_w * p.H + h) * D) + lane;
    const size_t step = static_cast<size_t>(p.H) * D / 4;
    for (int t0 = 0; t0 < T; t0 += 4) {
        float4 r[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (t0 + j < T)
                r[j] = src[(t0 + j) * step];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (t0 + j < T)
                *reinterpret_cast<float4 *>(si + (t0 + j) * SI_ROW + SI_V + 4 * lane) = r[j];
    }
}

// Stream 3: the forget gate d = exp(-5 sigmoid(raw_g)) per key channel and beta, four
// rows at a time with no branch around the arithmetic.
__device__ void gate_stream(const Layout &lay, const unsigned char *stg, float *si, float *sc, const Pre &pr, int T,
                            int lane)
{
    for (int t0 = 0; t0 < T; t0 += 4) {
        float4 dg[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 g = stage4(stg, lay, 3, min(t0 + j, T - 1), lane);
            dg[j] = make_float4(__expf(__fmul_rn(GATE_LOWER_BOUND, sigmoidf_(g.x))),
                                __expf(__fmul_rn(GATE_LOWER_BOUND, sigmoidf_(g.y))),
                                __expf(__fmul_rn(GATE_LOWER_BOUND, sigmoidf_(g.z))),
                                __expf(__fmul_rn(GATE_LOWER_BOUND, sigmoidf_(g.w))));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (t0 + j < T)
                store_perm(si + (t0 + j) * SI_ROW, 0, lane, dg[j]);
    }
    if (lane < T)
        sc[lane] = sigmoidf_(pr.beta);
}

// Each prologue warp also stages its stream's raw rows: item i's go to stage
// i % nstg, issued as soon as the warp is done with the stage's previous item, nstg
// items ahead.  The four prologue warps meet only at the scan-input buffers.
struct Stager {
    Item next;            // the item staged next
    bool pend0, pend1;    // a copy in flight into stage 0 / 1, for the drain on abort
    uint32_t par0, par1;  // and the phase parity that completes it
};

template <bool COLS, bool W, bool HR>
__device__ void prologue_warp(const ScanParams &p, const Layout &lay, unsigned char *sm, const Ctl &c, int n)
{
    const int pw = (threadIdx.x >> 5) - NSCAN, lane = threadIdx.x & 31;
    const uint32_t stg0 = smem_addr(sm + lay.stg(0));
    const uint32_t stage_bytes = static_cast<uint32_t>(lay.stg(1) - lay.stg(0));
    Pre pr;
    float4 win[3];  // the conv window carried from a unit's replay item into its verify item
    Item it = first_item(p, next_live(p, blockIdx.x, n, false), n);
    Stager sg{it, false, false, 0, 0};
    bool ok = true;
    int last_f = -1;  // the staged-rows flag this warp saw set last
    for (int b = 0; b < lay.nstg && sg.next.u < n; ++b) {  // the first nstg items' raw rows
        if (!rows_ready(p, c, sg.next.u, sg.next.part, lane, last_f)) {
            ok = false;
            break;
        }
        issue_stream<HR>(p, lay, stg0 + b * stage_bytes, c.bar(B_STG_FULL + 4 * b + pw), sg.next, pw, lane);
        (b ? sg.pend1 : sg.pend0) = true;
        sg.next = next_item(p, sg.next, n);
    }
    if (ok && it.u < n)
        load_pre<HR>(p, it, pw, lane, pr);
    for (int i = 0; ok && it.u < n; ++i) {
        const int b = i & 1;
        const Unit x = unit_of(p, it.u);
        const int T = it.part == 0 ? x.R : x.T;
        const int sb = lay.nstg == 2 ? b : 0, m = lay.nstg == 2 ? i >> 1 : i;
        const unsigned char *stg = sm + lay.stg(sb);
        if (!warp_wait(c, B_STG_FULL + 4 * sb + pw, m & 1)) {
            ok = false;
            break;
        }
        (sb ? sg.pend1 : sg.pend0) = false;
        if (HR && it.part == 1)
            copy_stage_out(p, lay, stg0 + sb * stage_bytes, it.u, pw, lane);
        // the scan of item i-2 has released this scan-input buffer
        if (i >= 2 && !warp_wait(c, B_SI_EMPTY + b, ((i >> 1) - 1) & 1)) {
            ok = false;
            break;
        }
        float *si = reinterpret_cast<float *>(sm + lay.si(b));
        float *sc = reinterpret_cast<float *>(sm + lay.sc(b));
        if (pw < 3) {
            if (it.part == 0 || x.R == 0) {  // a unit's first item starts from its ring
                win[0] = pr.ring[0];
                win[1] = pr.ring[1];
                win[2] = pr.ring[2];
            }
            // a replay ends in the committed ring (this round's ring snapshot)
            float *ring_dst = it.part == 0 ? p.ring_snap_out : p.ring_out;
            // an item without outputs never reads q-hat (the column stash still wants the
            // ring after every row); a replay with stored update vectors never reads v
            const bool stored_w = W && p.w_in && is_replay(p, it.part);
            if (!COLS && pw == 0 && (it.part == 0 || !p.out)) {
                roll_window(p, lay, stg, win, it.u, T, pw, lane, ring_dst);
            } else if (pw == 2 && stored_w) {
                copy_w_rows(p, si, it.u, T, lane);
                roll_window(p, lay, stg, win, it.u, T, pw, lane, ring_dst);
            } else {
                conv_stream<COLS>(p, lay, stg, si, pr.w, win, it.u, T, pw, lane, ring_dst);
            }
        } else {
            gate_stream(lay, stg, si, sc, pr, T, lane);
            if (HR && it.part == 1 && lane < p.T_rows) {  // the device copy of the raw beta
                const size_t bi = (static_cast<size_t>(x.lb) * p.T_rows + lane) * p.H + x.h;
                const uint32_t bits = __float_as_uint(pr.beta);  // bf16 widened exactly: its top half
                if (p.bf16)
                    static_cast<uint16_t *>(p.copy_beta)[bi] = static_cast<uint16_t>(bits >> 16);
                else
                    static_cast<uint32_t *>(p.copy_beta)[bi] = bits;
            }
        }
        mbar_arrive(c.bar(B_SI_FULL + b));
        // the raw rows of item i + nstg into the stage this warp is done with (before the
        // loads below: the proxy fence would wait for them), then the next item's conv
        // weights, ring and beta
        if (sg.next.u < n) {
            if (!rows_ready(p, c, sg.next.u, sg.next.part, lane, last_f)) {
                ok = false;
                break;
            }
            issue_stream<HR>(p, lay, stg0 + sb * stage_bytes, c.bar(B_STG_FULL + 4 * sb + pw), sg.next, pw, lane);
            (sb ? sg.pend1 : sg.pend0) = true;
            (sb ? sg.par1 : sg.par0) = (m + 1) & 1;
            sg.next = next_item(p, sg.next, n);
        }
        const Item nx = next_item(p, it, n);
        if (nx.u < n)
            load_pre<HR>(p, nx, pw, lane, pr);
        it = nx;
    }
    if (!ok && lane == 0) {  // stage copies in flight must land before the CTA leaves
        if (sg.pend0)
            drain_wait(c.bar(B_STG_FULL + pw), sg.par0);
        if (sg.pend1)
            drain_wait(c.bar(B_STG_FULL + 4 + pw), sg.par1);
    }
    if (HR) {  // this warp's copies: landed in, and sent out, before the CTA leaves
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (lane == 0)
            bulk_wait_all();
    }
}

// ---- scan warps ---------------------------------------------------------------------
// A thread's register tile to a [128][128] state at So (already offset by its columns):
// row rg + 8 r is the column pairs S[r][0], S[r][1], one 16-byte store.
__device__ __forceinline__ void store_tile(float *So, int rg, const float2 (&S)[16][2])
{
#pragma unroll
    for (int r = 0; r < 16; ++r)
        *reinterpret_cast<float4 *>(So + (rg + 8 * r) * D) = make_float4(S[r][0].x, S[r][0].y, S[r][1].x, S[r][1].y);
}

// The rows of one work item on the register tile S.  OUT: write the output rows to
// orow (lanes with b2 = 1, column jsum); without outputs (replays) neither e = S'^T q
// nor k.q is formed.  The state arithmetic, and so the state bits, do not depend on OUT.
template <bool COLS, bool OUT, bool W>
__device__ __forceinline__ void run_rows(const ScanParams &p, const float *si, const float *sc, float *orow,
                                         float *wrow, float2 (&S)[16][2], int T, int u, int rg, int cg, int jbase,
                                         int jsum, int b0, int b1, int b2)
{
    // ---- the T-row gated delta rule ---------------------------------------------
    for (int t = 0; t < T; ++t) {
        const float *vt = si + t * SI_ROW;
        const float *gp = vt + rg * GRP;
        float2 uacc[2], eacc[2];
        float2 kk2[16];  // (k, k) of each row, built once for both sweeps
        float kq = 0.f;  // k.q over this thread's 16 rows, in order (outputs only)
        uacc[0] = uacc[1] = eacc[0] = eacc[1] = make_float2(0.f, 0.f);
        // S' = d S ;  u = S'^T k ;  e = S'^T q   (this thread's 16 rows, in order)
#pragma unroll
        for (int rq = 0; rq < 4; ++rq) {
            const float4 d4 = *reinterpret_cast<const float4 *>(gp + 4 * rq);
            const float4 k4 = *reinterpret_cast<const float4 *>(gp + 16 + 4 * rq);
            const float4 q4 = *reinterpret_cast<const float4 *>(gp + 32 + 4 * rq);
            const float dv[4] = {d4.x, d4.y, d4.z, d4.w}, qv[4] = {q4.x, q4.y, q4.z, q4.w};
            const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
            if (OUT)
                kq = __fmaf_rn(k4.w, q4.w, __fmaf_rn(k4.z, q4.z, __fmaf_rn(k4.y, q4.y, __fmaf_rn(k4.x, q4.x, kq))));
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int r = 4 * rq + m;
                const float2 dd = make_float2(dv[m], dv[m]), kk = make_float2(kv[m], kv[m]);
                const float2 qq = make_float2(qv[m], qv[m]);
                kk2[r] = kk;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    S[r][h] = __fmul2_rn(S[r][h], dd);
                    uacc[h] = __ffma2_rn(S[r][h], kk, uacc[h]);
                    if (OUT)
                        eacc[h] = __ffma2_rn(S[r][h], qq, eacc[h]);
                }
            }
        }
        // reduce-scatter over the 8 row groups (lane bits 2..4): bits 3 and 2 split the 4
        // columns, then bit 4 splits u / e, so each sum ends on one lane; u is summed in
        // the same order with and without outputs (without, e is not carried at all)
        float sum;
        {
            // columns 0..3 of this thread: u in uacc, e in eacc; level 1 keeps columns
            // 2 b1, 2 b1 + 1 and sends the other two
            const float u0 = uacc[0].x, u1 = uacc[0].y, u2 = uacc[1].x, u3 = uacc[1].y;
            const float ua = __fadd_rn(b1 ? u2 : u0, __shfl_xor_sync(0xffffffffu, b1 ? u0 : u2, 8));
            const float ub = __fadd_rn(b1 ? u3 : u1, __shfl_xor_sync(0xffffffffu, b1 ? u1 : u3, 8));
            // level 2 keeps column 2 b1 + b0
            const float uc = __fadd_rn(b0 ? ub : ua, __shfl_xor_sync(0xffffffffu, b0 ? ua : ub, 4));
            if (OUT) {
                const float e0 = eacc[0].x, e1 = eacc[0].y, e2 = eacc[1].x, e3 = eacc[1].y;
                const float ea = __fadd_rn(b1 ? e2 : e0, __shfl_xor_sync(0xffffffffu, b1 ? e0 : e2, 8));
                const float eb = __fadd_rn(b1 ? e3 : e1, __shfl_xor_sync(0xffffffffu, b1 ? e1 : e3, 8));
                const float ec = __fadd_rn(b0 ? eb : ea, __shfl_xor_sync(0xffffffffu, b0 ? ea : eb, 4));
                // level 3: bit 4 splits u (b2 = 0) from e (b2 = 1)
                sum = __fadd_rn(b2 ? ec : uc, __shfl_xor_sync(0xffffffffu, b2 ? uc : ec, 16));
            } else {
                sum = __fadd_rn(uc, __shfl_xor_sync(0xffffffffu, uc, 16));
            }
        }
        if (OUT) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1)
                kq = __fadd_rn(kq, __shfl_xor_sync(0xffffffffu, kq, off));
        }
        // u lanes: w = beta (v - u); e lanes: o = (e + w (k.q)) / sqrt(128)
        const float beta = sc[t];
        const float w = __fmul_rn(beta, __fsub_rn(vt[SI_V + jsum], sum));
        // the u lanes (b2 = 0) hold w of column jsum: stored for a later replay
        if (W && wrow && !b2)
            wrow[static_cast<size_t>(t) * p.H * D] = w;
        const float w_of_col = __shfl_xor_sync(0xffffffffu, w, 16);
        // a warp's 16 e lanes store 16 consecutive columns of the output row
        if (OUT && b2)
            orow[static_cast<size_t>(t) * p.H * D] = __fmul_rn(__fmaf_rn(w_of_col, kq, sum), OUT_SCALE);
        // every lane gathers w of its 4 columns from the u lanes 4 c + cg
        float wv[4];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
            wv[c4] = __shfl_sync(0xffffffffu, w, 4 * c4 + cg);
        const float2 w01 = make_float2(wv[0], wv[1]), w23 = make_float2(wv[2], wv[3]);
        // S = S' + k w^T
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            S[r][0] = __ffma2_rn(kk2[r], w01, S[r][0]);
            S[r][1] = __ffma2_rn(kk2[r], w23, S[r][1]);
        }
        if (COLS)  // the column stash: the state after row t
            store_tile(p.s_cols + (static_cast<size_t>(u) * p.T_rows + t) * D * D + jbase, rg, S);
    }
}

// The rows of a replayed item whose update vectors the verify stored: per row
// S' = d S, then S = S' + k w^T with w_t read from the scan-input row.  These are the
// same two operations, on the same operands, that the verify applied to each element,
// so the state bits equal those of a replay that forms u and w again.
__device__ __forceinline__ void replay_rows_w(const float *si, float2 (&S)[16][2], int T, int rg, int jbase)
{
    for (int t = 0; t < T; ++t) {
        const float *vt = si + t * SI_ROW;
        const float *gp = vt + rg * GRP;
        const float4 w4 = *reinterpret_cast<const float4 *>(vt + SI_V + jbase);
        const float2 w01 = make_float2(w4.x, w4.y), w23 = make_float2(w4.z, w4.w);
#pragma unroll
        for (int rq = 0; rq < 4; ++rq) {
            const float4 d4 = *reinterpret_cast<const float4 *>(gp + 4 * rq);
            const float4 k4 = *reinterpret_cast<const float4 *>(gp + 16 + 4 * rq);
            const float dv[4] = {d4.x, d4.y, d4.z, d4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int r = 4 * rq + m;
                const float2 dd = make_float2(dv[m], dv[m]), kk = make_float2(kv[m], kv[m]);
                S[r][0] = __ffma2_rn(kk, w01, __fmul2_rn(S[r][0], dd));
                S[r][1] = __ffma2_rn(kk, w23, __fmul2_rn(S[r][1], dd));
            }
        }
    }
}

template <bool COLS, bool W>
__device__ void scan_warp(const ScanParams &p, const Layout &lay, unsigned char *sm, const Ctl &c, int n)
{
    // lane 4 rg + cg of warp wi holds key rows i = rg + 8 r (r < 16) of value columns
    // j = 16 wi + 4 cg + c (c < 4): 64 elements, column pairs (c, c + 1) packed, the
    // way they arrive from and leave for memory as 16-byte vectors.  The row scalars
    // d, k, q of a row are broadcast into both halves of a pair.  The two row groups
    // of a quarter warp read two addresses of a scan-input row, each broadcast to four
    // lanes.
    const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5, cg = lane & 3, rg = lane >> 2;
    const int jbase = 16 * wi + 4 * cg;
    // after the reduce-scatter a lane holds one sum: of u (b2 = 0) or e (b2 = 1), of
    // column jbase + 2 b1 + b0, where (b2, b1, b0) are the bits of rg
    const int b2 = (lane >> 4) & 1, b1 = (lane >> 3) & 1, b0 = (lane >> 2) & 1;
    const int jsum = jbase + 2 * b1 + b0;
    // this thread's 16-byte chunk of row rg in its box of the swizzled slot; row
    // rg + 8 r lies r * 1024 bytes further on with the same swizzle phase
    const uint32_t soff = (wi >> 1) * 16384 + rg * 128 + ((((wi & 1) * 4 + cg) ^ rg) << 4);
    // Scan warp 0 (the lead) also loads the states: unit k's into slot k % 2, two
    // units ahead, with the fused snapshot store leaving from the slot as soon as the
    // state has landed.  Its lane 0 reports invalid device keeps.
    const bool lead = wi == 0;
    const uint32_t slot0 = smem_addr(sm + lay.slot(0));
    constexpr uint32_t SLOT = D * D * 4;
    // lead: state copies in flight into slot 0 / 1, for the drain on abort, and the
    // phase parity that completes each
    bool pend0 = false, pend1 = false;
    uint32_t par0 = 0, par1 = 0;
    int u = next_live(p, blockIdx.x, n, lead && lane == 0);
    int u1 = u < n ? next_live(p, u + gridDim.x, n, lead && lane == 0) : n;
    int u2 = u1 < n ? next_live(p, u1 + gridDim.x, n, lead && lane == 0) : n;
    // the second unit's state is requested once the first has landed, so that the
    // first loads of all CTAs share the memory system with nothing else
    if (lead) {
        if (lane == 0 && u < n)
            issue_state(p, slot0, c.bar(B_STATE_FULL), u);
        pend0 = u < n;
    }
    bool ok = true;
    int i = 0;  // items through the scan-input buffers so far
    for (int k = 0; u < n; ++k) {
        const Unit x = unit_of(p, u);
        const int s = k & 1;
        const uint32_t ph = (k >> 1) & 1;
        if (!warp_wait(c, B_STATE_FULL + s, ph)) {
            ok = false;
            break;
        }
        if (lead) {
            (s ? pend1 : pend0) = false;
            if (k == 0 && u1 < n) {
                if (lane == 0)
                    issue_state(p, slot0 + SLOT, c.bar(B_STATE_FULL + 1), u1);
                pend1 = true;  // phase 0 of slot 1
            }
            if (p.s_snap && lane == 0) {
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    tma_store_2d(&p.tm_snap, 32 * b, u * D, slot0 + s * SLOT + b * 16384);
                bulk_commit();
            }
        }
        float2 S[16][2];  // S[r][h] = (S[rg + 8 r][jbase + 2 h], S[rg + 8 r][jbase + 2 h + 1])
        {
            const unsigned char *src = sm + lay.slot(s) + soff;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float4 a = *reinterpret_cast<const float4 *>(src + r * 1024);
                S[r][0] = make_float2(a.x, a.y);
                S[r][1] = make_float2(a.z, a.w);
            }
        }
        mbar_arrive(c.bar(B_STATE_EMPTY + s));
        // part 0: the replay of the previous round's kept rows (no outputs), after which
        // the state is this round's snapshot; part 1: this call's rows
        for (int part = x.R > 0 ? 0 : 1; part < 2; ++part, ++i) {
            const int T = part == 0 ? x.R : x.T;
            const int ib = i & 1;
            if (!warp_wait(c, B_SI_FULL + ib, (i >> 1) & 1)) {
                ok = false;
                break;
            }
            const float *si = reinterpret_cast<const float *>(sm + lay.si(ib));
            const float *sc = reinterpret_cast<const float *>(sm + lay.sc(ib));
            // the output row t of this unit: lanes with b2 = 1 store column jsum; the
            // update vectors of a verify item go to w_out (lanes with b2 = 0)
            float *orow = p.out && part == 1
                              ? p.out + (static_cast<size_t>(x.lb) * p.T_rows * p.H + x.h) * D + jsum
                              : nullptr;
            float *wrow = W && p.w_out && !is_replay(p, part)
                              ? p.w_out + (static_cast<size_t>(x.lb) * p.T_rows * p.H + x.h) * D + jsum
                              : nullptr;

            if (W && p.w_in && is_replay(p, part))
                replay_rows_w(si, S, T, rg, jbase);
            else if (orow)
                run_rows<COLS, true, W>(p, si, sc, orow, wrow, S, T, u, rg, cg, jbase, jsum, b0, b1, b2);
            else
                run_rows<COLS, false, W>(p, si, sc, orow, wrow, S, T, u, rg, cg, jbase, jsum, b0, b1, b2);
            mbar_arrive(c.bar(B_SI_EMPTY + ib));  // the scan inputs of item i are consumed
            if (part == 0)  // the committed state: this round's snapshot
                store_tile(p.s_snap_out + static_cast<size_t>(u) * D * D + jbase, rg, S);
        }
        if (!ok)
            break;

        // lead: every scan warp holds unit k in registers and the snapshot store has
        // read the slot: load unit k+2 into it
        if (lead && u2 < n) {
            if (!warp_wait(c, B_STATE_EMPTY + s, ph)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                bulk_wait_read();
                fence_proxy_async();
                issue_state(p, slot0 + s * SLOT, c.bar(B_STATE_FULL + s), u2);
            }
            (s ? pend1 : pend0) = true;
            (s ? par1 : par0) = ((k + 2) >> 1) & 1;
        }

        // ---- state write-back -----------------------------------------------------------
        store_tile(p.s_out + static_cast<size_t>(u) * D * D + jbase, rg, S);
        u = u1;
        u1 = u2;
        u2 = u2 < n ? next_live(p, u2 + gridDim.x, n, lead && lane == 0) : n;
    }
    if (lead && lane == 0) {
        if (!ok) {  // state copies in flight must land before the CTA leaves
            if (pend0)
                drain_wait(c.bar(B_STATE_FULL), par0);
            if (pend1)
                drain_wait(c.bar(B_STATE_FULL + 1), par1);
        }
        bulk_wait_all();  // the snapshot stores leave before the CTA's shared memory does
    }
}

// One persistent CTA per SM; warps 0..7 scan (warp 0 also loads the states), 8..11 run
// the prologue (warp 11 also stages the raw rows).
// COLS: also write the column stash (the state and ring after every row).  W: the
// verify stores each row's update vector (w_out) and a replay reads them (w_in); HR:
// this call's raw rows are read in place from host memory.  Each an instantiation of
// its own, so the launches without them carry none of their code.
// Verify and rollback share one instantiation: alternating between two kernels of this
// size cost the verify 5 % (its code is fetched again after each switch).
template <bool COLS, bool W, bool HR>
__global__ void __launch_bounds__(NT, 1) kda_scan_kernel(const __grid_constant__ ScanParams p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const Layout lay{p.tcap, p.bf16 ? 2 : 4, p.nstg};
    const Ctl c{smem_addr(sm + lay.bars()), reinterpret_cast<volatile int *>(sm + lay.flag()), p.status};
    const int n = p.L * p.B * p.H;  // below 2^31 / 128, checked at launch
    const int wi = threadIdx.x >> 5;
    // While the previous kernel finishes: L2 prefetches of the first two candidate
    // units' states (the buffer a replaying unit reads) and of the first unit's raw rows
    // of each stream, and the barrier set-up (shared memory only).
    if ((threadIdx.x & 31) == 0) {
        const int u0 = blockIdx.x, u1 = blockIdx.x + gridDim.x;
        if (wi == 0) {
            for (int b = 0; b < 4 && u0 < n; ++b)
                tma_prefetch_2d(&p.tm_in, 32 * b, u0 * D);
            for (int b = 0; b < 4 && u1 < n; ++b)
                tma_prefetch_2d(&p.tm_in, 32 * b, u1 * D);
        } else if (wi >= NSCAN && u0 < n) {
            const int lb = static_cast<int>(fdiv(static_cast<uint32_t>(u0), p.divH)), h = u0 - lb * p.H;
            if (!HR)
                tma_prefetch_4d(&p.tm_rows[wi - NSCAN], 0, h, 0, lb);
            if (p.keep_mode == DEFERRED)
                tma_prefetch_4d(&p.tm_prev[wi - NSCAN], 0, h, 0, lb);
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(c.bar(B_STATE_FULL + s), 1);
            mbar_init(c.bar(B_STATE_EMPTY + s), NSCAN * 32);
            mbar_init(c.bar(B_SI_FULL + s), NPRO * 32);
            mbar_init(c.bar(B_SI_EMPTY + s), NSCAN * 32);
        }
        for (int b = 0; b < 8; ++b)
            mbar_init(c.bar(B_STG_FULL + b), 1);
        *c.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // launched as a programmatic dependent: wait for the previous kernel's results.
    // The next kernel may be scheduled as soon as every CTA of this one is resident
    // (it waits for this kernel's results in turn).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (wi < NSCAN)
        scan_warp<COLS, W>(p, lay, sm, c, n);
    else
        prologue_warp<COLS, W, HR>(p, lay, sm, c, n);
}

// ---- host side ----------------------------------------------------------------------
using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiled lookup_encode()
{
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<EncodeTiled>(f);
}

// Tensor map of a state-shaped array [units * 128 rows][128] f32 with boxes of 32
// columns x 128 rows and the 128-byte swizzle.  Encoding is host-only; the last
// few maps of the calling thread are kept.
int state_map(CUtensorMap *m, const float *base, long long units)
{
    struct Entry {
        const float *base = nullptr;
        long long units = 0;
        CUtensorMap map;
    };
    thread_local Entry cache[4];
    thread_local int next = 0;
    for (const Entry &e : cache)
        if (e.base == base && e.units == units) {
            *m = e.map;
            return KDA_OK;
        }
    static const EncodeTiled encode = lookup_encode();
    if (!encode)
        return fail(KDA_ECUDA, "cuTensorMapEncodeTiled is not available from the CUDA driver");
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(units) * D};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * sizeof(float)};
    const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(D)};
    const cuuint32_t estr[2] = {1, 1};
    Entry &e = cache[next];
    const CUresult r = encode(&e.map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        e.base = nullptr;
        return fail(KDA_ECUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(static_cast<int>(r)));
    }
    e.base = base;
    e.units = units;
    next = (next + 1) % 4;
    *m = e.map;
    return KDA_OK;
}

// Tensor map of a raw-row tensor [LB][T_rows][H][128] (bf16 or f32) with boxes of one
// head's T_rows rows.  Encoding is host-only; the calling thread keeps the maps it
// encoded (cleared past 4096 entries).
int rows_map(CUtensorMap *m, const void *base, bool bf16, long long LB, int T_rows, int H)
{
    struct Key {
        const void *base;
        long long LB;
        int T_rows, H, bf16;
        bool operator==(const Key &o) const
        {
            return base == o.base && LB == o.LB && T_rows == o.T_rows && H == o.H && bf16 == o.bf16;
        }
    };
    struct Hash {
        size_t operator()(const Key &k) const
        {
            return std::hash<const void *>()(k.base) ^ (std::hash<long long>()(k.LB) * 31u) ^
                   (static_cast<size_t>(k.T_rows) << 20) ^ (static_cast<size_t>(k.H) << 8) ^ k.bf16;
        }
    };
    thread_local std::unordered_map<Key, CUtensorMap, Hash> cache;
    const Key key{base, LB, T_rows, H, bf16 ? 1 : 0};
    const auto it = cache.find(key);
    if (it != cache.end()) {
        *m = it->second;
        return KDA_OK;
    }
    static const EncodeTiled encode = lookup_encode();
    if (!encode)
        return fail(KDA_ECUDA, "cuTensorMapEncodeTiled is not available from the CUDA driver");
    const cuuint64_t es = bf16 ? 2 : 4;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(T_rows), static_cast<cuuint64_t>(LB)};
    const cuuint64_t strides[3] = {D * es, static_cast<cuuint64_t>(H) * D * es,
                                   static_cast<cuuint64_t>(T_rows) * H * D * es};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(D), 1, static_cast<cuuint32_t>(T_rows), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUtensorMap map;
    const CUresult r = encode(&map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(KDA_ECUDA, "cuTensorMapEncodeTiled (raw rows) failed with CUresult " +
                                   std::to_string(static_cast<int>(r)));
    if (cache.size() >= 4096)
        cache.clear();
    cache.emplace(key, map);
    *m = map;
    return KDA_OK;
}

struct DeviceInfo {
    std::atomic<int> ready{0};
    int sms = 0;
    int smem_max = 0;  // opt-in shared memory per block, set as the kernels' limit
};

// s_in: the state tm_in reads; for DEFERRED also s_in2 (tm_in2) and the previous
// round's raw rows.
FastDiv make_fastdiv(uint32_t d)
{
    uint32_t l = 0;
    while ((1ull << l) < d)
        ++l;
    const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
    return FastDiv{d, static_cast<uint32_t>(m), l};
}

int launch_scan(ScanParams &p, const float *s_in, cudaStream_t stream, const float *s_in2 = nullptr,
                const kda_rows *prev = nullptr, const kda_rows *copy = nullptr)
{
    const long long units = static_cast<long long>(p.L) * p.B * p.H;
    if (units == 0)
        return ok();
    if (units > 0x7fffffffLL / D)
        return fail(KDA_EINVAL, "L*B*H exceeds the unit index range (2^31 / 128 units)");
    p.divH = make_fastdiv(static_cast<uint32_t>(p.H));
    p.divB = make_fastdiv(static_cast<uint32_t>(p.B));
    static DeviceInfo info[64];
    static std::mutex init_mutex;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(KDA_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64)
        return fail(KDA_EINVAL, "device ordinal beyond the launch table");
    DeviceInfo &di = info[dev];
    if (!di.ready.load(std::memory_order_acquire)) {  // once per device, under a lock
        std::lock_guard<std::mutex> lock(init_mutex);
        if (!di.ready.load(std::memory_order_relaxed)) {
            int sms = 0, optin = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e == cudaSuccess)
                e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
            if (e != cudaSuccess)
                return fail(KDA_ECUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
            const size_t most = Layout{KDA_TMAX, 4, 1}.total();
            if (static_cast<size_t>(optin) < most)
                return fail(KDA_ECUDA,
                            "kda_scan_kernel needs " + std::to_string(most) + " bytes of shared memory per block");
            const void *kernels[5] = {reinterpret_cast<const void *>(kda_scan_kernel<false, false, false>),
                                      reinterpret_cast<const void *>(kda_scan_kernel<false, true, false>),
                                      reinterpret_cast<const void *>(kda_scan_kernel<true, false, false>),
                                      reinterpret_cast<const void *>(kda_scan_kernel<false, false, true>),
                                      reinterpret_cast<const void *>(kda_scan_kernel<false, true, true>)};
            for (const void *k : kernels)
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
            if (e != cudaSuccess)
                return fail(KDA_ECUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
            di.smem_max = optin;
            di.sms = sms;
            di.ready.store(1, std::memory_order_release);
        }
    }
    // two raw-row stages (the prologue then never waits for its rows) where they fit
    p.nstg = Layout{p.tcap, p.bf16 ? 2 : 4, 2}.total() <= static_cast<size_t>(di.smem_max) ? 2 : 1;
    const Layout lay{p.tcap, p.bf16 ? 2 : 4, p.nstg};
    int rc = state_map(&p.tm_in, s_in, units);
    if (rc)
        return rc;
    if (p.s_snap && (rc = state_map(&p.tm_snap, p.s_snap, units)))
        return rc;
    if (p.tcap < p.T_rows || (p.keep_mode == DEFERRED && p.tcap < p.T_prev))
        return fail(KDA_EINVAL, "internal: the raw-row stage must hold every round's rows");
    const long long LB = static_cast<long long>(p.L) * p.B;
    // rows in host memory are read with per-lane copies; their device copy has the maps
    const void *raw[4] = {p.xq, p.xk, p.xv, p.xg};
    if (p.rows_host && !copy)
        return fail(KDA_EINVAL, "internal: rows read in place need their device copy");
    const void *dst[4] = {copy ? copy->q : nullptr, copy ? copy->k : nullptr, copy ? copy->v : nullptr,
                          copy ? copy->g : nullptr};
    for (int s = 0; s < 4; ++s)
        if ((rc = p.rows_host ? rows_map(&p.tm_copy[s], dst[s], p.bf16 != 0, LB, p.T_rows, p.H)
                              : rows_map(&p.tm_rows[s], raw[s], p.bf16 != 0, LB, p.T_rows, p.H)))
            return rc;
    if (p.keep_mode == DEFERRED) {
        if (!s_in2 || !prev)
            return fail(KDA_EINVAL, "internal: a deferred round needs both state buffers and the previous rows");
        if ((rc = state_map(&p.tm_in2, s_in2, units)))
            return rc;
        const void *praw[4] = {prev->q, prev->k, prev->v, prev->g};
        for (int s = 0; s < 4; ++s)
            if ((rc = rows_map(&p.tm_prev[s], praw[s], p.bf16 != 0, LB, p.T_prev, p.H)))
                return rc;
    }
    const long long grid = std::min<long long>(units, di.sms);
    const unsigned g = static_cast<unsigned>(grid);
    const size_t sb = lay.total();
    // programmatic dependent launch: the kernel may be scheduled while the previous
    // kernel in the stream finishes; it waits for that kernel's results
    // (griddepcontrol.wait) before it touches global memory, so stream order holds
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(g);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = sb;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the column stash never carries update vectors (its rollback copies columns)
    const bool w = p.w_in || p.w_out;
    cudaError_t le;
    if (p.s_cols)
        le = cudaLaunchKernelEx(&cfg, kda_scan_kernel<true, false, false>, p);
    else if (p.rows_host)
        le = w ? cudaLaunchKernelEx(&cfg, kda_scan_kernel<false, true, true>, p)
               : cudaLaunchKernelEx(&cfg, kda_scan_kernel<false, false, true>, p);
    else
        le = w ? cudaLaunchKernelEx(&cfg, kda_scan_kernel<false, true, false>, p)
               : cudaLaunchKernelEx(&cfg, kda_scan_kernel<false, false, false>, p);
    if (le != cudaSuccess)
        return fail(KDA_ECUDA, std::string("kda_scan_kernel launch: ") + cudaGetErrorString(le));
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
    if (rows->w && !aligned16(rows->w))
        return fail(KDA_EINVAL, "rows->w (the update vectors) must be 16-byte aligned");
    return KDA_OK;
}

}  // namespace
}  // namespace kda

using namespace kda;
namespace kda {
namespace {

// Shared body of kda_verify_scan and kda_verify_scan_var.  t_rows == nullptr: every
// session runs T rows; else session b runs t_rows[b] rows (host or device values).
// pingpong: the pre-round state and ring are read from the stash (left untouched, so
// they are the round's snapshot) and the post-round ones written to st.
int verify_common(const kda_dims *dims, const kda_layer_state *st, const kda_rows *rows, int T,
                  const int *t_rows, int t_mem, float *out, kda_stash *stash, int *dev_status, bool pingpong,
                  cudaStream_t stream)
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
    if (pingpong && !stash)
        return fail(KDA_EINVAL, "kda_verify_scan_pingpong needs a stash holding the pre-round state and ring");
    if (stash) {
        if (!stash->state_snap || !stash->ring_snap)
            return fail(KDA_EINVAL, "stash->state_snap and stash->ring_snap must be allocated by the caller");
        if (!aligned16(stash->state_snap) || !aligned16(stash->ring_snap))
            return fail(KDA_EINVAL, "stash snapshots must be 16-byte aligned");
        if (stash->state_snap == st->state || stash->ring_snap == st->conv_ring)
            return fail(KDA_EINVAL, "the snapshots must not alias the resident state");
    }
    ScanParams p{};
    p.keep_mode = KEEP_NONE;
    if (t_rows) {
        if (t_mem == KDA_MEM_HOST) {
            if (dims->B > KDA_HOST_KEEP_MAX)
                return fail(KDA_EINVAL, "B exceeds KDA_HOST_KEEP_MAX for host row counts; pass them on the device");
            for (int b = 0; b < dims->B; ++b) {
                if (t_rows[b] < 1 || t_rows[b] > T)
                    return fail(KDA_EINVAL, "t_rows[" + std::to_string(b) + "] = " + std::to_string(t_rows[b]) +
                                                " outside 1.." + std::to_string(T));
                p.keep_host[b] = static_cast<unsigned char>(t_rows[b]);
            }
            p.keep_mode = ROWS_HOST;
        } else if (t_mem == KDA_MEM_DEVICE) {
            if (reinterpret_cast<uintptr_t>(t_rows) & 3u)
                return fail(KDA_EINVAL, "device t_rows must be 4-byte aligned");
            p.keep_mode = ROWS_DEVICE;
            p.rows_dev = t_rows;
        } else {
            return fail(KDA_EINVAL, "t_mem must be KDA_MEM_HOST or KDA_MEM_DEVICE");
        }
    }
    p.s_out = st->state;
    p.s_snap = stash && !pingpong ? stash->state_snap : nullptr;
    p.ring_in = pingpong ? stash->ring_snap : st->conv_ring;
    p.ring_out = st->conv_ring;
    p.ring_snap = stash && !pingpong ? stash->ring_snap : nullptr;
    p.conv_w = st->conv_w;
    p.xq = rows->q; p.xk = rows->k; p.xv = rows->v; p.xg = rows->g; p.xb = rows->beta;
    p.w_out = rows->w;
    p.out = out;
    p.status = dev_status;
    p.L = dims->L; p.B = dims->B; p.H = dims->H;
    p.T_rows = T;
    p.T_run = T;
    p.tcap = T;
    p.bf16 = dims->dtype == KDA_BF16;
    if ((rc = launch_scan(p, pingpong ? stash->state_snap : st->state, stream)))
        return rc;
    if (stash) {
        stash->rows = *rows;
        stash->T = T;
    }
    return ok();
}

}  // namespace
}  // namespace kda

extern "C" int kda_verify_scan(const kda_dims *dims, const kda_layer_state *st, const kda_rows *rows,
                               int T, float *out, kda_stash *stash, cudaStream_t stream)
{
    return verify_common(dims, st, rows, T, nullptr, KDA_MEM_HOST, out, stash, nullptr, false, stream);
}

extern "C" int kda_verify_scan_var(const kda_dims *dims, const kda_layer_state *st, const kda_rows *rows,
                                   int T_cap, const int *t_rows, int t_mem, float *out, kda_stash *stash,
                                   int *dev_status, cudaStream_t stream)
{
    if (!t_rows && dims && static_cast<long long>(dims->L) * dims->B * dims->H > 0)
        return fail(KDA_EINVAL, "t_rows must not be NULL");
    return verify_common(dims, st, rows, T_cap, t_rows, t_mem, out, stash, dev_status, false, stream);
}

extern "C" int kda_verify_scan_pingpong(const kda_dims *dims, const kda_layer_state *st, const kda_rows *rows,
                                        int T, const int *t_rows, int t_mem, float *out, kda_stash *stash,
                                        int *dev_status, cudaStream_t stream)
{
    return verify_common(dims, st, rows, T, t_rows, t_mem, out, stash, dev_status, true, stream);
}

namespace kda {
namespace {

// The device address of each raw-row pointer of host rows (pinned host memory mapped
// into the device's address space), checked like device rows.
int host_rows_on_device(const kda_rows *host_rows, int dtype, kda_rows *dev)
{
    int rc = check_rows(host_rows, dtype);
    if (rc)
        return rc;
    const void *h[5] = {host_rows->q, host_rows->k, host_rows->v, host_rows->g, host_rows->beta};
    void *d[5];
    for (int i = 0; i < 5; ++i)
        if (cudaHostGetDevicePointer(&d[i], const_cast<void *>(h[i]), 0) != cudaSuccess) {
            cudaGetLastError();
            return fail(KDA_EINVAL, "host_rows must be pinned host memory the device can address "
                                    "(cudaHostGetDevicePointer refused one of them)");
        }
    *dev = kda_rows{d[0], d[1], d[2], d[3], d[4], nullptr};
    return check_rows(dev, dtype);
}

// Shared body of kda_verify_scan_deferred, kda_verify_scan_deferred_staged (ready:
// nullptr for rows already in place) and kda_verify_scan_deferred_host (host_rows: this
// call's rows read in place from host memory, `rows` their device copy).
int deferred_common(const kda_dims *dims, kda_layer_state *st, kda_stash *stash, const int *prev_keep,
                    const kda_rows *rows, int T, float *out, const unsigned *ready, int ppf, unsigned epoch,
                    int *dev_status, cudaStream_t stream, const kda_rows *host_rows = nullptr)
{
    int rc = check_common(dims, st);
    if (rc)
        return rc;
    if (!stash)
        return fail(KDA_EINVAL, "kda_verify_scan_deferred needs the stash of the previous ping-pong round");
    if (T < 1 || T > KDA_TMAX)
        return fail(KDA_EINVAL, "T must lie in 1..15 (K <= 14 drafts per round), got " + std::to_string(T));
    if (stash->T < 1 || stash->T > KDA_TMAX)
        return fail(KDA_EINVAL, "stash->T is not a verify round's row count (run a ping-pong verify first)");
    const bool empty = static_cast<long long>(dims->L) * dims->B * dims->H == 0;
    if (!empty) {
        if ((rc = check_rows(rows, dims->dtype)) || (rc = check_rows(&stash->rows, dims->dtype)))
            return rc;
        if (!stash->state_snap || !stash->ring_snap || !aligned16(stash->state_snap) || !aligned16(stash->ring_snap))
            return fail(KDA_EINVAL, "stash snapshots must be non-NULL and 16-byte aligned");
        if (stash->state_snap == st->state || stash->ring_snap == st->conv_ring)
            return fail(KDA_EINVAL, "the two state buffers (and the two ring buffers) must be distinct");
        if (!prev_keep || (reinterpret_cast<uintptr_t>(prev_keep) & 3u))
            return fail(KDA_EINVAL, "prev_keep must be a 4-byte aligned device array of B ints");
        if (out && (reinterpret_cast<uintptr_t>(out) & 3u))
            return fail(KDA_EINVAL, "out must be 4-byte aligned");
        kda_rows hdev{};
        if (host_rows && (rc = host_rows_on_device(host_rows, dims->dtype, &hdev)))
            return rc;
        ScanParams p{};
        p.keep_mode = DEFERRED;
        p.keep_dev = prev_keep;
        p.T_prev = stash->T;
        // P (the stash's buffers): the previous round's pre-round state, replayed from,
        // then this round's post-round state; Q (st's buffers): the previous round's
        // post-round state, then this round's snapshot
        p.s_out = stash->state_snap;
        p.s_snap_out = st->state;
        p.ring_in = stash->ring_snap;
        p.ring_in2 = st->conv_ring;
        p.ring_out = stash->ring_snap;
        p.ring_snap_out = st->conv_ring;
        p.conv_w = st->conv_w;
        p.xq = rows->q; p.xk = rows->k; p.xv = rows->v; p.xg = rows->g; p.xb = rows->beta;
        if (host_rows) {  // read in place; `rows` receives their device copy
            p.xq = hdev.q; p.xk = hdev.k; p.xv = hdev.v; p.xg = hdev.g; p.xb = hdev.beta;
            p.copy_beta = const_cast<void *>(rows->beta);
            p.rows_host = 1;
        }
        p.xb_prev = stash->rows.beta;
        p.w_out = rows->w;
        p.w_in = stash->rows.w;
        p.T_w = stash->T;
        if (p.w_out && p.w_out == p.w_in)
            return fail(KDA_EINVAL, "rows->w must not be the previous round's update vectors (stash->rows.w)");
        p.out = out;
        p.status = dev_status;
        p.L = dims->L; p.B = dims->B; p.H = dims->H;
        p.T_rows = T;
        p.T_run = T;
        p.tcap = std::max(T, stash->T);
        p.bf16 = dims->dtype == KDA_BF16;
        p.ready = ready;
        p.ready_ppf = ppf;
        p.epoch = epoch;
        if ((rc = launch_scan(p, stash->state_snap, stream, st->state, &stash->rows, host_rows ? rows : nullptr)))
            return rc;
    }
    // the stash now describes this round (its snapshot is in Q) and st its post-round
    // state (in P): the buffers exchange roles
    std::swap(st->state, stash->state_snap);
    std::swap(st->conv_ring, stash->ring_snap);
    stash->rows = rows ? *rows : kda_rows{};
    stash->T = T;
    return ok();
}

}  // namespace
}  // namespace kda

extern "C" int kda_verify_scan_deferred(const kda_dims *dims, kda_layer_state *st, kda_stash *stash,
                                        const int *prev_keep, const kda_rows *rows, int T, float *out,
                                        int *dev_status, cudaStream_t stream)
{
    return kda::deferred_common(dims, st, stash, prev_keep, rows, T, out, nullptr, 1, 0, dev_status, stream);
}

extern "C" int kda_verify_scan_deferred_staged(const kda_dims *dims, kda_layer_state *st, kda_stash *stash,
                                               const int *prev_keep, const kda_rows *rows, int T, float *out,
                                               const unsigned *ready_flags, int pairs_per_flag, unsigned epoch,
                                               int *dev_status, cudaStream_t stream)
{
    if (!ready_flags || (reinterpret_cast<uintptr_t>(ready_flags) & 3u))
        return kda::fail(KDA_EINVAL, "ready_flags must be a 4-byte aligned device array of flags");
    if (pairs_per_flag < 1)
        return kda::fail(KDA_EINVAL, "pairs_per_flag must be >= 1");
    return kda::deferred_common(dims, st, stash, prev_keep, rows, T, out, ready_flags, pairs_per_flag, epoch,
                                dev_status, stream);
}

extern "C" int kda_verify_scan_deferred_host(const kda_dims *dims, kda_layer_state *st, kda_stash *stash,
                                             const int *prev_keep, const kda_rows *host_rows, const kda_rows *rows,
                                             int T, float *out, int *dev_status, cudaStream_t stream)
{
    if (!host_rows)
        return kda::fail(KDA_EINVAL, "host_rows must not be NULL");
    return kda::deferred_common(dims, st, stash, prev_keep, rows, T, out, nullptr, 1, 0, dev_status, stream,
                                host_rows);
}

namespace kda {
namespace {

// *flag = value in stream order, by the stream (cuStreamWriteValue32 from the driver)
int write_flag(unsigned *flag, unsigned value, cudaStream_t stream)
{
    using WriteValue = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
    static const WriteValue write = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<WriteValue>(nullptr);
        return reinterpret_cast<WriteValue>(f);
    }();
    if (!write)
        return fail(KDA_ECUDA, "cuStreamWriteValue32 is not available from the CUDA driver");
    const CUresult r = write(reinterpret_cast<CUstream>(stream), reinterpret_cast<CUdeviceptr>(flag), value,
                             CU_STREAM_WRITE_VALUE_DEFAULT);
    if (r != CUDA_SUCCESS)
        return fail(KDA_ECUDA, "cuStreamWriteValue32 failed with CUresult " + std::to_string(static_cast<int>(r)));
    return KDA_OK;
}

}  // namespace
}  // namespace kda

extern "C" int kda_stream_write_u32(unsigned *flag, unsigned value, cudaStream_t stream)
{
    if (!flag || (reinterpret_cast<uintptr_t>(flag) & 3u))
        return kda::fail(KDA_EINVAL, "flag must be a 4-byte aligned device pointer");
    const int rc = kda::write_flag(flag, value, stream);
    return rc ? rc : kda::ok();
}

extern "C" int kda_upload_rows_staged(const kda_dims *dims, const kda_rows *dst, const kda_rows *src, int T,
                                      unsigned *ready_flags, int pairs_per_flag, unsigned epoch,
                                      cudaStream_t stream)
{
    if (!dims || !dst || !src)
        return kda::fail(KDA_EINVAL, "dims, dst and src must not be NULL");
    if (dims->L < 0 || dims->B < 0 || dims->H < 0)
        return kda::fail(KDA_EINVAL, "L, B, H must be >= 0");
    if (dims->dtype != KDA_F32 && dims->dtype != KDA_BF16)
        return kda::fail(KDA_EINVAL, "dtype must be KDA_F32 or KDA_BF16");
    if (T < 1 || T > KDA_TMAX)
        return kda::fail(KDA_EINVAL, "T must lie in 1..15, got " + std::to_string(T));
    if (!ready_flags || (reinterpret_cast<uintptr_t>(ready_flags) & 3u))
        return kda::fail(KDA_EINVAL, "ready_flags must be a 4-byte aligned device array of flags");
    if (pairs_per_flag < 1)
        return kda::fail(KDA_EINVAL, "pairs_per_flag must be >= 1");
    const void *d[5] = {dst->q, dst->k, dst->v, dst->g, dst->beta};
    const void *h[5] = {src->q, src->k, src->v, src->g, src->beta};
    const size_t es = dims->dtype == KDA_BF16 ? 2 : 4;
    const int pairs = dims->L * dims->B;  // (layer, session) pairs, lb = l B + b
    const size_t per_pair = static_cast<size_t>(T) * dims->H * es;  // beta; x128 for q, k, v, g
    if (per_pair == 0 || pairs == 0)
        return kda::ok();
    for (int i = 0; i < 5; ++i)
        if (!d[i] || !h[i])
            return kda::fail(KDA_EINVAL, "every raw-row pointer of dst and src must be non-NULL");
    // q, k, v, g at one distance from each other on both sides (one allocation of four
    // equal tensors): a range of pairs of all four is one 2D copy (four rows of the range's
    // bytes, pitch that distance), since the copy engine pays for every copy
    const auto gap = [](const void *a, const void *b) {
        return static_cast<long long>(reinterpret_cast<uintptr_t>(b)) -
               static_cast<long long>(reinterpret_cast<uintptr_t>(a));
    };
    const size_t tensor_bytes = per_pair * D * pairs;
    const long long dp = gap(d[0], d[1]), hp = gap(h[0], h[1]);
    const long long max_pitch = 0x7fffffffLL;  // the copy engine's pitch limit, and then some
    bool two_d = dp >= static_cast<long long>(tensor_bytes) && hp >= static_cast<long long>(tensor_bytes) &&
                       dp <= max_pitch && hp <= max_pitch &&
                       gap(d[1], d[2]) == dp && gap(d[2], d[3]) == dp && gap(h[1], h[2]) == hp &&
                       gap(h[2], h[3]) == hp;
    for (int p0 = 0, f = 0; p0 < pairs; p0 += pairs_per_flag, ++f) {
        const int n = std::min(pairs_per_flag, pairs - p0);
        for (int i = 0; i < 5; ++i) {
            const size_t row = i < 4 ? per_pair * D : per_pair;
            char *dd = static_cast<char *>(const_cast<void *>(d[i])) + row * p0;
            const char *hh = static_cast<const char *>(h[i]) + row * p0;
            cudaError_t e;
            if (two_d && i == 0) {
                // the runtime checks the whole span: four tensors of separate allocations
                // are refused before anything is queued, and then go one by one
                e = cudaMemcpy2DAsync(dd, static_cast<size_t>(dp), hh, static_cast<size_t>(hp), row * n, 4,
                                      cudaMemcpyHostToDevice, stream);
                if (e == cudaSuccess) {
                    i = 3;  // q, k, v and g are done
                    continue;
                }
                cudaGetLastError();
                two_d = false;
            }
            e = cudaMemcpyAsync(dd, hh, row * n, cudaMemcpyHostToDevice, stream);
            if (e != cudaSuccess)
                return kda::fail(KDA_ECUDA, std::string("cudaMemcpyAsync: ") + cudaGetErrorString(e));
        }
        const int rc = kda::write_flag(ready_flags + f, epoch, stream);
        if (rc)
            return rc;
    }
    return kda::ok();
}

namespace kda {
namespace {

// Shared body of kda_rollback and kda_rollback_var.  t_rows == nullptr: the round ran
// stash->T rows for every session; else t_rows[b] rows for session b (same memory kind
// as keep).
int rollback_common(const kda_dims *dims, const kda_layer_state *st, const kda_stash *stash, const int *t_rows,
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
            const int tb = t_rows ? t_rows[b] : stash->T;
            if (tb < 1 || tb > stash->T)
                return fail(KDA_EINVAL, "t_rows[" + std::to_string(b) + "] = " + std::to_string(tb) + " outside 1.." +
                                            std::to_string(stash->T));
            if (keep[b] < 1 || keep[b] > tb)
                return fail(KDA_EINVAL, "keep[" + std::to_string(b) + "] = " + std::to_string(keep[b]) +
                                            " outside 1.." + std::to_string(tb) +
                                            " (the anchor row is always kept; keep = accepted drafts + 1)");
            // a session that keeps all of its rows has nothing to restore
            p.keep_host[b] = static_cast<unsigned char>(keep[b] < tb ? keep[b] : stash->T);
            any |= keep[b] < tb;
        }
        if (!any)
            return ok();
        p.keep_mode = KEEP_HOST;
    } else if (keep_mem == KDA_MEM_DEVICE) {
        if ((reinterpret_cast<uintptr_t>(keep) & 3u) || (reinterpret_cast<uintptr_t>(t_rows) & 3u))
            return fail(KDA_EINVAL, "device keep and t_rows must be 4-byte aligned");
        p.keep_mode = KEEP_DEVICE;
        p.keep_dev = keep;
        p.rows_dev = t_rows;
    } else {
        return fail(KDA_EINVAL, "keep_mem must be KDA_MEM_HOST or KDA_MEM_DEVICE");
    }
    p.s_out = st->state;
    p.s_snap = nullptr;
    p.ring_in = stash->ring_snap;
    p.ring_out = st->conv_ring;
    p.ring_snap = nullptr;
    p.conv_w = st->conv_w;
    p.xq = stash->rows.q; p.xk = stash->rows.k; p.xv = stash->rows.v;
    p.xg = stash->rows.g; p.xb = stash->rows.beta;
    p.w_in = stash->rows.w;
    p.T_w = stash->T;
    p.out = nullptr;
    p.status = dev_status;
    p.L = dims->L; p.B = dims->B; p.H = dims->H;
    p.T_rows = stash->T;
    p.T_run = stash->T;
    p.tcap = stash->T;
    p.bf16 = dims->dtype == KDA_BF16;
    return launch_scan(p, stash->state_snap, stream);
}

}  // namespace
}  // namespace kda

extern "C" int kda_rollback(const kda_dims *dims, const kda_layer_state *st, const kda_stash *stash,
                            const int *keep, int keep_mem, int *dev_status, cudaStream_t stream)
{
    return rollback_common(dims, st, stash, nullptr, keep, keep_mem, dev_status, stream);
}

extern "C" int kda_rollback_var(const kda_dims *dims, const kda_layer_state *st, const kda_stash *stash,
                                const int *t_rows, const int *keep, int mem, int *dev_status, cudaStream_t stream)
{
    if (!t_rows && dims && static_cast<long long>(dims->L) * dims->B * dims->H > 0)
        return fail(KDA_EINVAL, "t_rows must not be NULL");
    return rollback_common(dims, st, stash, t_rows, keep, mem, dev_status, stream);
}

// ---------------------------------------------------------------------------
// Column-stash rollback (the alternative the pages weigh against snapshot + replay:
// vLLM keeps num_spec + 1 state columns and commits the accepted one).  The verify
// writes the state and conv ring after every row; rollback copies the kept column.
// ---------------------------------------------------------------------------
namespace kda {
namespace {

// One CTA per unit: state <- state_cols[keep-1], ring <- ring_cols[keep-1] for the
// units of sessions that keep fewer than all rows.
__global__ void __launch_bounds__(256) commit_cols_kernel(const __grid_constant__ ScanParams p)
{
    const int n = p.L * p.B * p.H;
    for (int u = blockIdx.x; u < n; u += gridDim.x) {
        const int kp = unit_rows(p, (u / p.H) % p.B);
        if (kp < 0 && p.status && threadIdx.x == 0)
            atomicOr(p.status, KDA_ST_BADKEEP);
        if (kp <= 0)
            continue;
        const float4 *src = reinterpret_cast<const float4 *>(p.s_cols + (static_cast<size_t>(u) * p.T_rows + kp - 1) * D * D);
        float4 *dst = reinterpret_cast<float4 *>(p.s_out + static_cast<size_t>(u) * D * D);
        for (int i = threadIdx.x; i < D * D / 4; i += blockDim.x)
            dst[i] = src[i];
        const float4 *rsrc =
            reinterpret_cast<const float4 *>(p.ring_cols + (static_cast<size_t>(u) * p.T_rows + kp - 1) * 9 * D);
        float4 *rdst = reinterpret_cast<float4 *>(p.ring_out + static_cast<size_t>(u) * 9 * D);
        for (int i = threadIdx.x; i < 9 * D / 4; i += blockDim.x)
            rdst[i] = rsrc[i];
    }
}

}  // namespace
}  // namespace kda

extern "C" int kda_verify_scan_cols(const kda_dims *dims, const kda_layer_state *st, const kda_rows *rows, int T,
                                    float *out, float *state_cols, float *ring_cols, cudaStream_t stream)
{
    int rc = check_common(dims, st);
    if (rc)
        return rc;
    if (T < 1 || T > KDA_TMAX)
        return fail(KDA_EINVAL, "T must lie in 1..15 (K <= 14 drafts per round), got " + std::to_string(T));
    if (static_cast<long long>(dims->L) * dims->B * dims->H == 0)
        return ok();
    if ((rc = check_rows(rows, dims->dtype)))
        return rc;
    if (out && (reinterpret_cast<uintptr_t>(out) & 3u))
        return fail(KDA_EINVAL, "out must be 4-byte aligned");
    if (!state_cols || !ring_cols || !aligned16(state_cols) || !aligned16(ring_cols))
        return fail(KDA_EINVAL, "state_cols and ring_cols must be 16-byte aligned device memory");
    ScanParams p{};
    p.keep_mode = KEEP_NONE;
    p.s_out = st->state;
    p.ring_in = st->conv_ring;
    p.ring_out = st->conv_ring;
    p.conv_w = st->conv_w;
    p.xq = rows->q; p.xk = rows->k; p.xv = rows->v; p.xg = rows->g; p.xb = rows->beta;
    p.out = out;
    p.s_cols = state_cols;
    p.ring_cols = ring_cols;
    p.L = dims->L; p.B = dims->B; p.H = dims->H;
    p.T_rows = T;
    p.T_run = T;
    p.tcap = T;
    p.bf16 = dims->dtype == KDA_BF16;
    return launch_scan(p, st->state, stream);
}

extern "C" int kda_rollback_cols(const kda_dims *dims, const kda_layer_state *st, const float *state_cols,
                                 const float *ring_cols, int T, const int *keep, int keep_mem, int *dev_status,
                                 cudaStream_t stream)
{
    int rc = check_common(dims, st);
    if (rc)
        return rc;
    if (T < 1 || T > KDA_TMAX)
        return fail(KDA_EINVAL, "T must lie in 1..15, got " + std::to_string(T));
    const long long units = static_cast<long long>(dims->L) * dims->B * dims->H;
    if (units == 0)
        return ok();
    if (!state_cols || !ring_cols || !aligned16(state_cols) || !aligned16(ring_cols))
        return fail(KDA_EINVAL, "state_cols and ring_cols must be 16-byte aligned device memory");
    if (!keep)
        return fail(KDA_EINVAL, "keep must not be NULL");
    ScanParams p{};
    if (keep_mem == KDA_MEM_HOST) {
        if (dims->B > KDA_HOST_KEEP_MAX)
            return fail(KDA_EINVAL, "B exceeds KDA_HOST_KEEP_MAX for a host keep array; pass keep on the device");
        bool any = false;
        for (int b = 0; b < dims->B; ++b) {
            if (keep[b] < 1 || keep[b] > T)
                return fail(KDA_EINVAL, "keep[" + std::to_string(b) + "] = " + std::to_string(keep[b]) +
                                            " outside 1.." + std::to_string(T));
            p.keep_host[b] = static_cast<unsigned char>(keep[b]);
            any |= keep[b] < T;
        }
        if (!any)
            return ok();
        p.keep_mode = KEEP_HOST;
    } else if (keep_mem == KDA_MEM_DEVICE) {
        if (reinterpret_cast<uintptr_t>(keep) & 3u)
            return fail(KDA_EINVAL, "device keep must be 4-byte aligned");
        p.keep_mode = KEEP_DEVICE;
        p.keep_dev = keep;
    } else {
        return fail(KDA_EINVAL, "keep_mem must be KDA_MEM_HOST or KDA_MEM_DEVICE");
    }
    p.s_out = st->state;
    p.ring_out = st->conv_ring;
    p.s_cols = const_cast<float *>(state_cols);
    p.ring_cols = const_cast<float *>(ring_cols);
    p.status = dev_status;
    p.L = dims->L; p.B = dims->B; p.H = dims->H;
    p.T_rows = T;
    p.T_run = T;
    p.bf16 = dims->dtype == KDA_BF16;
    const long long grid = std::min<long long>(units, 4096);  // a grid-stride loop over the units
    commit_cols_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(p);
    return check_launch("commit_cols_kernel");
}
