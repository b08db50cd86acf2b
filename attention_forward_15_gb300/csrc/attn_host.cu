// attn_fwd_host: the forward for inputs and outputs in host memory, pipelined
// over chunks of heads so that the copies of both directions and the kernels
// overlap.  Host code only; it reaches the device through the library's own
// public entry points (attn_fwd_check, attn_fwd_plan, attn_fwd_work, attn_fwd)
// and the CUDA runtime's copies, streams and events.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "attn.h"

namespace {

constexpr int kMaxDevices = 64;

// Per device: the copy-in and copy-out streams beside the caller's, and the
// events that order the three (created on the first call on that device).
struct HostPipe {
    int sms = 0;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev_start = nullptr, ev_in = nullptr, ev_out = nullptr, ev_end = nullptr;
};

std::mutex g_pipe_mutex;   // one call's copy/launch sequence at a time
HostPipe g_pipe[kMaxDevices];

// The B*H heads are cut into chunks that flow through three stages at once:
// chunk c+1's inputs are copied in while chunk c is computed and chunk c-1's
// outputs are copied out.  Measured on GB300 with page-locked host buffers, the
// CPU-GPU link moves about 207 GB/s in or 190 GB/s out in one direction, about
// 260 GB/s in total with both active, each copy costs about 2.2 us more, and
// the forward's rate per SM is about 4.4, 7.8 and 11.9 TFLOP/s with the
// kernels that run D <= 64, D <= 128 and D <= 256.  With n equal chunks the
// pipeline takes
//   first chunk's copy in
//   + max(link time of every other copy, forwards of all chunks but the last)
//   + last chunk's forward and copy out,
// a forward taking whole waves of its chunk's work units.  Few chunks pay long
// ends; many pay more copies and emptier waves.
constexpr int kMaxHostChunks = 16;
constexpr double kInBytesPerUs = 207e3, kOutBytesPerUs = 190e3, kBothBytesPerUs = 260e3, kCopyUs = 2.2;

double host_kernel_us(int heads, int L, int D, int mask_kind, int block_size, int sms) {
    double flops = 0.0;
    int units = 0;
    if (attn_fwd_work(1, heads, L, D, mask_kind, block_size, ATTN_F16, &flops, nullptr) != ATTN_OK ||
        attn_fwd_plan(1, heads, L, D, mask_kind, block_size, ATTN_F16, &units, nullptr, nullptr, nullptr) !=
            ATTN_OK ||
        units <= 0)
        return 0.0;
    const double waves = std::ceil(static_cast<double>(units) / sms);
    const double rate_sm = D <= 64 ? 4.4e6 : (D <= 128 ? 7.8e6 : 11.9e6);   // flops per us per SM
    return waves * (flops / units) / rate_sm + 4.0;
}

double host_pipeline_us(int BH, int hc, int L, int D, int mask_kind, int block_size, int sms) {
    const int n = (BH + hc - 1) / hc;
    const int last = BH - (n - 1) * hc;
    const double in_head = 3.0 * L * D * 2.0, out_head = static_cast<double>(L) * (D * 2.0 + 4.0);
    const double head = hc * in_head / kInBytesPerUs + 3 * kCopyUs;
    const double link_rest = ((BH - hc) * in_head + (BH - last) * out_head) / kBothBytesPerUs +
                             5 * (n - 1) * kCopyUs;
    const double k_full = host_kernel_us(hc, L, D, mask_kind, block_size, sms);
    const double k_last = host_kernel_us(last, L, D, mask_kind, block_size, sms);
    const double tail = k_last + last * out_head / kOutBytesPerUs + 2 * kCopyUs;
    return head + std::max(link_rest, (n - 1) * k_full) + tail;
}

// Heads per chunk (the last chunk may hold fewer).  A chunk's lse slice starts
// hc * L floats in and must stay 16-byte aligned, so for L not a multiple of 4
// a chunk holds a multiple of 4 / gcd(L, 4) heads.
int host_heads_per_chunk(int BH, int L, int D, int mask_kind, int block_size, int sms) {
    const int m = L % 4 == 0 ? 1 : (L % 2 == 0 ? 2 : 4);
    int best = BH;
    double best_t = host_pipeline_us(BH, BH, L, D, mask_kind, block_size, sms);
    for (int n = 2; n <= kMaxHostChunks && n <= BH; ++n) {
        int hc = (BH + n - 1) / n;
        hc = (hc + m - 1) / m * m;
        if (hc >= BH) continue;
        const double t = host_pipeline_us(BH, hc, L, D, mask_kind, block_size, sms);
        if (t < best_t) {
            best_t = t;
            best = hc;
        }
    }
    return best;
}

char *at(const void *p, size_t off) { return const_cast<char *>(static_cast<const char *>(p)) + off; }

}  // namespace

extern "C" {

int attn_fwd_host_chunks(int B, int H, int L, int D, int mask_kind, int block_size, int dtype, int sms,
                         int *heads_per_chunk, int *chunks) {
    // shape checks only (placeholder buffers: an empty problem passes before
    // any pointer is looked at, and a non-empty one gets 16-aligned stand-ins)
    const bool empty = static_cast<long long>(B) * H * L == 0;
    void *stand_in = empty ? nullptr : reinterpret_cast<void *>(static_cast<uintptr_t>(16));
    int rc = attn_fwd_check(stand_in, stand_in, stand_in, stand_in, nullptr, B, H, L, D, mask_kind,
                            block_size, 1.0f, dtype);
    if (rc != ATTN_OK) return rc;
    if (sms <= 0) return ATTN_ERR_ARG;
    int hc = 0, n = 0;
    if (!empty) {
        const int bh = B * H;
        hc = host_heads_per_chunk(bh, L, D, mask_kind, block_size, sms);
        n = (bh + hc - 1) / hc;
    }
    if (heads_per_chunk) *heads_per_chunk = hc;
    if (chunks) *chunks = n;
    return ATTN_OK;
}

int attn_fwd_host(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h,
                  void *q_d, void *k_d, void *v_d, void *o_d, float *lse_d, int B, int H, int L,
                  int D, int mask_kind, int block_size, float sm_scale, int dtype, void *stream) {
    // the device buffers get attn_fwd's checks (shape, scale, null, alignment)
    int rc = attn_fwd_check(q_d, k_d, v_d, o_d, lse_h ? lse_d : nullptr, B, H, L, D, mask_kind, block_size,
                            sm_scale, dtype);
    if (rc != ATTN_OK) return rc;
    if (static_cast<long long>(B) * H * L == 0) return ATTN_OK;   // empty problem
    if (!q_h || !k_h || !v_h || !o_h || (lse_h && !lse_d)) return ATTN_ERR_NULL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int BH = B * H;
    const size_t head_bytes = static_cast<size_t>(L) * D * 2;
    const size_t head_lse = static_cast<size_t>(L);
    {
        std::lock_guard<std::mutex> lk(g_pipe_mutex);
        HostPipe &p = g_pipe[dev];
        if (!p.h2d) {
            if (cudaDeviceGetAttribute(&p.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) != cudaSuccess ||
                cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) != cudaSuccess ||
                cudaEventCreateWithFlags(&p.ev_start, cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&p.ev_in, cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&p.ev_out, cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&p.ev_end, cudaEventDisableTiming) != cudaSuccess) {
                p.h2d = nullptr;   // retried on the next call
                return ATTN_ERR_CUDA;
            }
        }
        const int hc = host_heads_per_chunk(BH, L, D, mask_kind, block_size, p.sms);
        // both copy streams start after the work already queued on the caller's
        // stream (which may still use the device buffers)
        if (cudaEventRecord(p.ev_start, s) != cudaSuccess ||
            cudaStreamWaitEvent(p.h2d, p.ev_start, 0) != cudaSuccess ||
            cudaStreamWaitEvent(p.d2h, p.ev_start, 0) != cudaSuccess)
            return ATTN_ERR_CUDA;
        // A wait takes the event's record at the time of the call, so each
        // record, followed at once by its wait, can reuse the one event.
        for (int h0 = 0; h0 < BH && rc == ATTN_OK; h0 += hc) {
            const int n = std::min(hc, BH - h0);
            const size_t off = h0 * head_bytes, bytes = n * head_bytes;
            if (cudaMemcpyAsync(at(q_d, off), at(q_h, off), bytes, cudaMemcpyHostToDevice, p.h2d) != cudaSuccess ||
                cudaMemcpyAsync(at(k_d, off), at(k_h, off), bytes, cudaMemcpyHostToDevice, p.h2d) != cudaSuccess ||
                cudaMemcpyAsync(at(v_d, off), at(v_h, off), bytes, cudaMemcpyHostToDevice, p.h2d) != cudaSuccess ||
                cudaEventRecord(p.ev_in, p.h2d) != cudaSuccess || cudaStreamWaitEvent(s, p.ev_in, 0) != cudaSuccess) {
                rc = ATTN_ERR_CUDA;
                break;
            }
            float *lse_c = lse_h ? lse_d + h0 * head_lse : nullptr;
            rc = attn_fwd(at(q_d, off), at(k_d, off), at(v_d, off), at(o_d, off), lse_c, 1, n, L, D, mask_kind,
                          block_size, sm_scale, dtype, stream);
            if (rc != ATTN_OK) break;
            if (cudaEventRecord(p.ev_out, s) != cudaSuccess || cudaStreamWaitEvent(p.d2h, p.ev_out, 0) != cudaSuccess ||
                cudaMemcpyAsync(at(o_h, off), at(o_d, off), bytes, cudaMemcpyDeviceToHost, p.d2h) != cudaSuccess ||
                (lse_h && cudaMemcpyAsync(lse_h + h0 * head_lse, lse_c, n * head_lse * sizeof(float),
                                          cudaMemcpyDeviceToHost, p.d2h) != cudaSuccess))
                rc = ATTN_ERR_CUDA;
        }
        // the caller's stream waits for both copy streams, also after a failure,
        // so that neither stays forked from it
        if (cudaEventRecord(p.ev_end, p.h2d) != cudaSuccess || cudaStreamWaitEvent(s, p.ev_end, 0) != cudaSuccess ||
            cudaEventRecord(p.ev_end, p.d2h) != cudaSuccess || cudaStreamWaitEvent(s, p.ev_end, 0) != cudaSuccess)
            rc = rc == ATTN_OK ? ATTN_ERR_CUDA : rc;
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
    return rc;
}

}  // extern "C"
