// kda_round.cpp -- one speculative round driven from host memory in one call: the
// round's raw rows, logits and drafts go up from pinned host buffers, the verify runs
// (folding in the previous round's accept), the accept runs, and j and the bonus come
// back to the host.  glm_spec.rs, glm5_spec_round: a round is draft, verify, accept and
// rollback, and the next round's drafts follow from this round's accept, so the host
// waits for j every round.  This file issues the library's own entry points in stream
// order; it launches no kernel of its own.

#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <climits>
#include <string>

#include "kda_internal.h"
#include "kda_spec.h"

namespace {

constexpr int KDA_JB_PENDING = INT_MIN;  // no j or bonus takes this value

// The host-to-device copy of a raw-row set: one copy per tensor (q, k, v, g, beta).
int upload_rows(const kda_dims *dims, const kda_rows *dst, const kda_rows *src, int T, cudaStream_t s)
{
    const size_t es = dims->dtype == KDA_BF16 ? 2 : 4;
    const size_t beta = static_cast<size_t>(dims->L) * dims->B * T * dims->H * es;
    const size_t bytes = beta * KDA_DK;
    const void *d[5] = {dst->q, dst->k, dst->v, dst->g, dst->beta};
    const void *h[5] = {src->q, src->k, src->v, src->g, src->beta};
    for (int i = 0; i < 5; ++i) {
        if (!d[i] || !h[i])
            return kda::fail(KDA_EINVAL, "every raw-row pointer of dev_rows and host_rows must be non-NULL");
        const cudaError_t e = cudaMemcpyAsync(const_cast<void *>(d[i]), h[i], i < 4 ? bytes : beta,
                                              cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess)
            return kda::fail(KDA_ECUDA, std::string("cudaMemcpyAsync: ") + cudaGetErrorString(e));
    }
    return KDA_OK;
}

int copy(void *dst, const void *src, size_t bytes, cudaMemcpyKind kind, cudaStream_t s)
{
    if (bytes == 0)
        return KDA_OK;
    const cudaError_t e = cudaMemcpyAsync(dst, src, bytes, kind, s);
    if (e != cudaSuccess)
        return kda::fail(KDA_ECUDA, std::string("cudaMemcpyAsync: ") + cudaGetErrorString(e));
    return KDA_OK;
}

}  // namespace

extern "C" int kda_round_host(const kda_dims *dims, kda_layer_state *st, kda_stash *stash, int T,
                              const kda_rows *host_rows, const kda_rows *dev_rows, const void *host_logits,
                              void *dev_logits, int logit_dtype, int V, const int *host_drafts, int *dev_drafts,
                              int *dev_jbk, int *host_jb, float *out, unsigned *ready_flags, int pairs_per_flag,
                              unsigned epoch, int *dev_status, cudaStream_t stream, cudaStream_t copy_stream,
                              int rows_in_place, int wait)
{
    if (!dims || !st || !stash || !host_rows || !dev_rows)
        return kda::fail(KDA_EINVAL, "dims, st, stash, host_rows and dev_rows must not be NULL");
    if (!host_logits || !dev_logits || !host_drafts || !dev_drafts || !dev_jbk || !host_jb)
        return kda::fail(KDA_EINVAL, "the logits, drafts and result buffers must not be NULL");
    if (dims->B < 0 || dims->L < 0 || dims->H < 0)
        return kda::fail(KDA_EINVAL, "L, B, H must be >= 0");
    if (T < 1 || T > KDA_TMAX)
        return kda::fail(KDA_EINVAL, "T must lie in 1..15, got " + std::to_string(T));
    if (V < 1)
        return kda::fail(KDA_EINVAL, "V must be >= 1");
    if (logit_dtype != KDA_F32 && logit_dtype != KDA_BF16)
        return kda::fail(KDA_EINVAL, "logit_dtype must be KDA_F32 or KDA_BF16");
    if (reinterpret_cast<uintptr_t>(dev_jbk) & 3u)
        return kda::fail(KDA_EINVAL, "dev_jbk must be a 4-byte aligned device array [3][B]");
    if (stream == copy_stream && stash->T > 0 && !rows_in_place)
        return kda::fail(KDA_EINVAL, "copy_stream must differ from stream (the copies overlap the verify)");
    const int B = dims->B;
    int *j_out = dev_jbk, *bonus_out = dev_jbk + B, *keep = dev_jbk + 2 * B;
    const size_t logit_bytes = static_cast<size_t>(B) * T * V * (logit_dtype == KDA_BF16 ? 2 : 4);
    const size_t draft_bytes = static_cast<size_t>(B) * (T - 1) * sizeof(int);
    int rc;
    if (stash->T == 0) {
        // the first round of a chain: the raw rows go up whole, then a ping-pong verify
        if ((rc = upload_rows(dims, dev_rows, host_rows, T, stream)) ||
            (rc = copy(dev_logits, host_logits, logit_bytes, cudaMemcpyHostToDevice, stream)) ||
            (rc = copy(dev_drafts, host_drafts, draft_bytes, cudaMemcpyHostToDevice, stream)))
            return rc;
        // st receives the post-round state, the stash keeps the pre-round state and
        // records the rows: the pair as the next (deferred) round wants it
        if ((rc = kda_verify_scan_pingpong(dims, st, dev_rows, T, nullptr, KDA_MEM_HOST, out, stash, dev_status,
                                           stream)))
            return rc;
    } else if (rows_in_place) {
        // the verify reads the rows in place from host memory and leaves their device
        // copy in dev_rows; the logits and drafts go up meanwhile
        if ((rc = kda_verify_scan_deferred_host(dims, st, stash, keep, host_rows, dev_rows, T, out, dev_status,
                                                stream)))
            return rc;
        if ((rc = copy(dev_logits, host_logits, logit_bytes, cudaMemcpyHostToDevice, copy_stream)) ||
            (rc = copy(dev_drafts, host_drafts, draft_bytes, cudaMemcpyHostToDevice, copy_stream)))
            return rc;
        cudaEvent_t copied;
        cudaError_t e = cudaEventCreateWithFlags(&copied, cudaEventDisableTiming);
        if (e == cudaSuccess) {
            e = cudaEventRecord(copied, copy_stream);
            if (e == cudaSuccess)
                e = cudaStreamWaitEvent(stream, copied, 0);
            cudaEventDestroy(copied);
        }
        if (e != cudaSuccess)
            return kda::fail(KDA_ECUDA, std::string("cudaStreamWaitEvent: ") + cudaGetErrorString(e));
    } else {
        // the launch first (its start-up overlaps the first range's copy; it scans each
        // range once its flag is set), then the rows by range of pairs_per_flag (layer,
        // session) pairs with their ready flags, then the logits and drafts, which the
        // accept waits for
        if ((rc = kda_verify_scan_deferred_staged(dims, st, stash, keep, dev_rows, T, out, ready_flags,
                                                  pairs_per_flag, epoch, dev_status, stream)))
            return rc;
        // the launch has been queued: from here a refused copy leaves it waiting on a flag
        // until its one-second bound, which then sets KDA_ST_TIMEOUT
        if ((rc = kda_upload_rows_staged(dims, dev_rows, host_rows, T, ready_flags, pairs_per_flag, epoch,
                                         copy_stream)) ||
            (rc = copy(dev_logits, host_logits, logit_bytes, cudaMemcpyHostToDevice, copy_stream)) ||
            (rc = copy(dev_drafts, host_drafts, draft_bytes, cudaMemcpyHostToDevice, copy_stream)))
            return rc;
        // (an event destroyed while pending is released once it completes)
        cudaEvent_t copied;
        cudaError_t e = cudaEventCreateWithFlags(&copied, cudaEventDisableTiming);
        if (e == cudaSuccess) {
            e = cudaEventRecord(copied, copy_stream);
            if (e == cudaSuccess)
                e = cudaStreamWaitEvent(stream, copied, 0);
            cudaEventDestroy(copied);
        }
        if (e != cudaSuccess)
            return kda::fail(KDA_ECUDA, std::string("cudaStreamWaitEvent: ") + cudaGetErrorString(e));
    }
    // j and the bonus: written by the accept straight into host_jb where the device can
    // address it (pinned memory mapped into the device's address space), else copied
    // back after it; keep stays on the device for the next round's verify
    void *mapped = nullptr;
    if (cudaHostGetDevicePointer(&mapped, host_jb, 0) != cudaSuccess) {
        cudaGetLastError();  // not mapped: the copy below
        mapped = nullptr;
    }
    int *jo = mapped ? static_cast<int *>(mapped) : j_out, *bo = mapped ? static_cast<int *>(mapped) + B : bonus_out;
    // mapped and waited for: the results are awaited by reading host_jb until the
    // accept has replaced a value no result takes (the stream's earlier work was waited
    // for by the previous call, or is ordered before this accept)
    const bool poll = mapped && wait;
    if (poll)
        for (int i = 0; i < 2 * B; ++i)
            reinterpret_cast<volatile int *>(host_jb)[i] = KDA_JB_PENDING;
    if ((rc = spec_accept(dev_logits, logit_dtype, B, T, V, dev_drafts, jo, bo, keep, dev_status, nullptr, 0,
                          stream)))
        return rc;
    if (!mapped &&
        (rc = copy(host_jb, dev_jbk, 2 * static_cast<size_t>(B) * sizeof(int), cudaMemcpyDeviceToHost, stream)))
        return rc;
    if (poll) {
        // spin on the mapped results (a second at most, then the stream's own wait,
        // which also reports a failed launch)
        const volatile int *r = host_jb;
        const auto t0 = std::chrono::steady_clock::now();
        for (int i = 0; i < 2 * B;) {
            if (r[i] != KDA_JB_PENDING) {
                ++i;
                continue;
            }
            if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(1))
                break;
        }
        std::atomic_thread_fence(std::memory_order_acquire);
    }
    if (wait) {
        const cudaError_t e = poll ? cudaStreamQuery(stream) : cudaStreamSynchronize(stream);
        if (e != cudaSuccess && e != cudaErrorNotReady)
            return kda::fail(KDA_ECUDA, std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e));
        if (poll && e == cudaErrorNotReady) {
            cudaGetLastError();
            for (int i = 0; i < 2 * B; ++i)
                if (host_jb[i] == KDA_JB_PENDING) {  // the accept has not written: wait for the stream
                    const cudaError_t e2 = cudaStreamSynchronize(stream);
                    if (e2 != cudaSuccess)
                        return kda::fail(KDA_ECUDA, std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e2));
                    break;
                }
        }
    }
    return kda::ok();
}
