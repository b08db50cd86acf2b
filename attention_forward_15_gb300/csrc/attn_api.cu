// Host side of the C ABI declared in include/attn.h: argument validation,
// TMA tensor-map encoding, kernel selection and launch.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "attn.h"
#include "attn_bwd_kernel.cuh"
#include "attn_fwd_kernel.cuh"

namespace {

using attn::Cfg;
using attn::FwdParams;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int sms = 0;
    unsigned int *status = nullptr;   // device status word written by timed-out waits
    bool smem_attr[9][2] = {};        // per (kernel, dtype): dynamic smem attribute set
    bool bwd_attr[3][2][2] = {};      // backward: per (head dim, dtype, dK/dV | dQ)
    // backward: a second stream for the dQ kernel, forked from and joined back
    // into the caller's stream by two events (created on the first backward)
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

std::mutex g_mutex;
std::mutex g_bwd_mutex;   // one backward's fork/launch/join sequence at a time
DeviceState g_dev[kMaxDevices];
int g_inject = 0;   // fault-injection mode for the next attn_fwd calls (tests only)
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Head dims: any multiple of 8 from 8 to 256.  Kernels exist for 64, 128 and
// 256; a smaller head dim runs in the next one up, its tensor maps declaring
// the true width so that the missing columns load as zeros (they add nothing to
// Q K^T and give zero columns of O, which are not stored).
bool head_dim_ok(int D) { return D >= 8 && D <= 256 && D % 8 == 0; }
int kernel_dim(int D) { return D <= 64 ? 64 : (D <= 128 ? 128 : 256); }
int head_dim_index(int D) { return kernel_dim(D) == 64 ? 0 : (kernel_dim(D) == 128 ? 1 : 2); }
// Block-diagonal with blocks of at most 64 keys: every key tile is masked and
// a row attends one 64-key half of it (the one-half instantiations).
bool small_blocks(int mask_kind, int block_size) {
    return mask_kind == ATTN_MASK_BLOCK_DIAG && block_size <= 64;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape/argument validation shared by every entry point (no CUDA calls).
int validate_shape(int B, int H, int L, int D, int mask_kind, int block_size, int dtype) {
    if (B < 0 || H < 0 || L < 0) return ATTN_ERR_SHAPE;
    if (mask_kind < ATTN_MASK_DENSE || mask_kind > ATTN_MASK_BLOCK_DIAG) return ATTN_ERR_UNSUPPORTED;
    if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
    if (!head_dim_ok(D)) return ATTN_ERR_UNSUPPORTED;
    if (mask_kind == ATTN_MASK_BLOCK_DIAG) {
        if (block_size <= 0) return ATTN_ERR_BLOCK_SIZE;
        if (L > 0 && L % block_size != 0) return ATTN_ERR_BLOCK_SIZE;
        if (!(block_size % attn::BN == 0 || attn::BN % block_size == 0)) return ATTN_ERR_UNSUPPORTED;
    }
    // element counts must stay addressable and TMA dimensions within 2^32
    const long long bh = static_cast<long long>(B) * H;
    if (bh > 0x7fffffffLL) return ATTN_ERR_SHAPE;
    const long long elems = bh * L * static_cast<long long>(D);
    if (elems > (1LL << 46)) return ATTN_ERR_SHAPE;
    return ATTN_OK;
}

struct Plan {
    bool pair;
    int n_qt, n_kv, n_units;
};

Plan make_plan(int B, int H, int L, int D) {
    Plan pl;
    pl.pair = kernel_dim(D) <= 128;
    pl.n_qt = (L + attn::BM - 1) / attn::BM;
    pl.n_kv = (L + attn::BN - 1) / attn::BN;
    const int per_bh = pl.pair ? (pl.n_qt + 1) / 2 : pl.n_qt;
    pl.n_units = B * H * per_bh;
    return pl;
}

// K and V of the whole problem comfortably inside the 129 MB L2: every query
// tile of a head re-reads its K/V, so asking L2 to keep them pays.
bool kv_fits_l2(int BH, int L, int D) {
    return 2.0 * BH * static_cast<double>(L) * D * 2.0 <= 64.0 * 1024 * 1024;
}

int threads_for(int D) {
    switch (kernel_dim(D)) {
        case 64: return Cfg<64, true>::THREADS;
        case 128: return Cfg<128, true>::THREADS;
        default: return Cfg<256, false>::THREADS;
    }
}

int smem_for(int D) {
    switch (kernel_dim(D)) {
        case 64: return Cfg<64, true>::SMEM_BYTES;
        case 128: return Cfg<128, true>::SMEM_BYTES;
        default: return Cfg<256, false>::SMEM_BYTES;
    }
}

int load_encoder() {
    if (g_encode) return ATTN_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return ATTN_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return ATTN_OK;
}

// Per-device state: SM count and the status word (allocated once per device).
int device_state(DeviceState **out, int *dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mutex);
    int rc = load_encoder();
    if (rc != ATTN_OK) return rc;
    DeviceState &st = g_dev[dev];
    if (!st.ready) {
        if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        if (cudaMalloc(&st.status, sizeof(unsigned int)) != cudaSuccess) return ATTN_ERR_CUDA;
        if (cudaMemset(st.status, 0, sizeof(unsigned int)) != cudaSuccess) return ATTN_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
        st.ready = true;
    }
    *out = &st;
    if (dev_out) *dev_out = dev;
    return ATTN_OK;
}

// 3-D tensor map over a [BH, L, D] 16-bit array: box = 64 columns (128 bytes)
// x `rows` rows (128; 64 for the half-tile ring entries of the D = 256
// backward; 32 for the forward's staged O stores) x 1 head, 128-byte swizzle;
// rows past L read as zero (and are not written by stores).
int encode_map(CUtensorMap *m, const void *ptr, int BH, int L, int D, int dtype, int rows = 128) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                             static_cast<cuuint64_t>(L) * static_cast<cuuint64_t>(D) * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          3, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// 3-D tensor map over a [BH, L, D] 16-bit output for the backward's stores:
// box = 32 columns (64 bytes) x 32 rows x 1 head, 64-byte swizzle; the part of
// a box past L or D is not written.
int encode_store_map(CUtensorMap *m, const void *ptr, int BH, int L, int D, int dtype) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                             static_cast<cuuint64_t>(L) * static_cast<cuuint64_t>(D) * 2};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          3, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// 3-D tensor map over V^T as float8 e5m2 bytes, [BH, D, L] with keys innermost:
// box = 128 keys (128 bytes) x `rows` head-dim rows, 128-byte swizzle; rows
// past D read as zero.
int encode_map_vt8(CUtensorMap *m, const void *ptr, int BH, int L, int D, int rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(D),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(L),
                             static_cast<cuuint64_t>(L) * static_cast<cuuint64_t>(D)};
    cuuint32_t box[3] = {128, static_cast<cuuint32_t>(rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// BDH: the block-diagonal instantiation for blocks of at most 64 keys (D <= 128,
// 16-bit P), chosen by the callers below.
template <int D, bool BF16, bool PAIR, bool FP8V = false, bool BDH = false>
int launch(DeviceState &st, const void *q, const void *k, const void *v, FwdParams prm, int dtype,
           cudaStream_t stream) {
    static_assert(!BDH || (D <= 128 && !FP8V), "one-half block-diagonal kernels: D <= 128, 16-bit P");
    using C = Cfg<D, PAIR, FP8V>;
    auto kern = attn::attn_fwd_kernel<D, BF16, PAIR, FP8V, BDH>;
    {
        std::lock_guard<std::mutex> lk(g_mutex);
        bool &set = st.smem_attr[head_dim_index(D) + (FP8V ? 3 : 0) + (BDH ? 6 : 0)][BF16 ? 1 : 0];
        if (!set) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::SMEM_BYTES) != cudaSuccess)
                return ATTN_ERR_CUDA;
            if constexpr (C::REGSPLIT) {
                // The kernel moves registers between warpgroups (setmaxnreg); the
                // split assumes the block's pool is THREADS x REGS_LAUNCH.  A
                // smaller pool would leave the increase waiting forever, so such a
                // build is refused here rather than launched.
                cudaFuncAttributes fa;
                if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return ATTN_ERR_CUDA;
                if (fa.numRegs != C::REGS_LAUNCH) return ATTN_ERR_UNSUPPORTED;
            }
            set = true;
        }
    }
    CUtensorMap tq, tk, tv, to;
    std::memset(&to, 0, sizeof(to));      // (unused unless O rows are staged)
    int rc = encode_map(&tq, q, prm.BH, prm.L, prm.d_out, dtype);
    if (rc == ATTN_OK) rc = encode_map(&tk, k, prm.BH, prm.L, prm.d_out, dtype);
    if (rc == ATTN_OK)
        rc = FP8V ? encode_map_vt8(&tv, v, prm.BH, prm.L, prm.d_out, D / C::EPT)
                  : encode_map(&tv, v, prm.BH, prm.L, prm.d_out, dtype);
    if (rc == ATTN_OK && C::OSTAGE) rc = encode_map(&to, prm.o, prm.BH, prm.L, prm.d_out, dtype, 32);
    if (rc != ATTN_OK) return rc;
    const int grid = prm.n_units < st.sms ? prm.n_units : st.sms;
    // Programmatic dependent launch: the CTAs may be scheduled while the
    // previous kernel of the stream finishes; the kernel waits for that
    // kernel's completion (griddepcontrol.wait) before its first global access.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, to, prm) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

int attn_abi_version(void) { return (1 << 16) | 1; }

int attn_debug_inject(int mode) {
    if (mode != 0 && mode != 1) return ATTN_ERR_ARG;
    g_inject = mode;
    return ATTN_OK;
}

const char *attn_status_string(int status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_NULL: return "null pointer";
        case ATTN_ERR_SHAPE: return "bad shape";
        case ATTN_ERR_BLOCK_SIZE: return "block size must be positive and divide L";
        case ATTN_ERR_UNSUPPORTED: return "unsupported head dim, dtype, mask kind or block size";
        case ATTN_ERR_ALIGN: return "pointer not 16-byte aligned";
        case ATTN_ERR_CUDA: return "CUDA error";
        case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
        case ATTN_ERR_ARG: return "bad argument";
        default: return "unknown status";
    }
}

int attn_fwd_work(int B, int H, int L, int D, int mask_kind, int block_size, int dtype,
                  double *flops, double *bytes) {
    int rc = validate_shape(B, H, L, D, mask_kind, block_size, dtype);
    if (rc != ATTN_OK) return rc;
    const double bh = static_cast<double>(B) * H;
    const double Ld = L;
    double pairs;
    if (mask_kind == ATTN_MASK_DENSE)
        pairs = Ld * Ld;
    else if (mask_kind == ATTN_MASK_CAUSAL)
        pairs = Ld * (Ld + 1.0) / 2.0;
    else
        pairs = Ld * block_size;
    if (flops) *flops = 4.0 * D * pairs * bh;
    if (bytes) *bytes = 4.0 * bh * Ld * D * 2.0;
    return ATTN_OK;
}

int attn_fwd_plan(int B, int H, int L, int D, int mask_kind, int block_size, int dtype, int *units,
                  int *ctas, int *threads, int *smem_bytes) {
    int rc = validate_shape(B, H, L, D, mask_kind, block_size, dtype);
    if (rc != ATTN_OK) return rc;
    const Plan pl = make_plan(B, H, L, D);
    if (units) *units = pl.n_units;
    if (threads) *threads = threads_for(D);
    if (smem_bytes) *smem_bytes = smem_for(D);
    if (ctas) {
        int sms = 0, dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        *ctas = pl.n_units < sms ? pl.n_units : sms;
    }
    return ATTN_OK;
}

}  // extern "C"

namespace {

// The host-side checks of a forward call (attn_fwd, attn_fwd_noalloc,
// attn_fwd_fp8v with FP8V): no CUDA call and no access to the buffers.
// *launch is set to false for an empty problem (nothing to enqueue).
template <bool FP8V>
int check_fwd_args(const void *q, const void *k, const void *v, const void *o, const void *lse, int B,
                   int H, int L, int D, int mask_kind, int block_size, float sm_scale, int dtype,
                   bool *launch) {
    *launch = false;
    int rc = validate_shape(B, H, L, D, mask_kind, block_size, dtype);
    if (rc != ATTN_OK) return rc;
    if (!std::isfinite(sm_scale)) return ATTN_ERR_ARG;
    // V^T rows are L bytes: TMA needs them to be a multiple of 16 bytes
    if (FP8V && L % 16 != 0) return ATTN_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * H * L == 0) return ATTN_OK;   // empty problem
    if (!q || !k || !v || !o) return ATTN_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
        return ATTN_ERR_ALIGN;
    *launch = true;
    return ATTN_OK;
}

// attn_fwd and attn_fwd_fp8v: validation, plan, parameters and the launch of the
// kernel for the head dim (FP8V: V given as e5m2 V^T).
template <bool FP8V>
int fwd_common(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int L,
               int D, int mask_kind, int block_size, float sm_scale, int dtype, void *stream) {
    bool go = false;
    int rc = check_fwd_args<FP8V>(q, k, v, o, lse, B, H, L, D, mask_kind, block_size, sm_scale, dtype, &go);
    if (rc != ATTN_OK || !go) return rc;

    DeviceState *st = nullptr;
    rc = device_state(&st, nullptr);
    if (rc != ATTN_OK) return rc;

    const Plan pl = make_plan(B, H, L, D);
    FwdParams prm;
    prm.o = o;
    prm.lse = lse;
    prm.status = st->status;
    prm.BH = B * H;
    prm.L = L;
    prm.mask = mask_kind;
    prm.bs = mask_kind == ATTN_MASK_BLOCK_DIAG ? block_size : 0;
    prm.n_qt = pl.n_qt;
    prm.n_kv = pl.n_kv;
    prm.n_units = pl.n_units;
    prm.scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634074);
    prm.inject = g_inject;
    prm.kv_keep = kv_fits_l2(prm.BH, L, D) ? 1 : 0;
    prm.d_out = D;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool bf16 = dtype == ATTN_BF16;
    if constexpr (!FP8V) {
        if (small_blocks(mask_kind, block_size) && kernel_dim(D) <= 128)
            return kernel_dim(D) == 64 ? (bf16 ? launch<64, true, true, false, true>(*st, q, k, v, prm, dtype, s)
                                               : launch<64, false, true, false, true>(*st, q, k, v, prm, dtype, s))
                                       : (bf16 ? launch<128, true, true, false, true>(*st, q, k, v, prm, dtype, s)
                                               : launch<128, false, true, false, true>(*st, q, k, v, prm, dtype, s));
    }
    switch (kernel_dim(D)) {
        case 64:
            return bf16 ? launch<64, true, true, FP8V>(*st, q, k, v, prm, dtype, s)
                        : launch<64, false, true, FP8V>(*st, q, k, v, prm, dtype, s);
        case 128:
            return bf16 ? launch<128, true, true, FP8V>(*st, q, k, v, prm, dtype, s)
                        : launch<128, false, true, FP8V>(*st, q, k, v, prm, dtype, s);
        default:
            return bf16 ? launch<256, true, false, FP8V>(*st, q, k, v, prm, dtype, s)
                        : launch<256, false, false, FP8V>(*st, q, k, v, prm, dtype, s);
    }
}

}  // namespace

extern "C" {

int attn_fwd_check(const void *q, const void *k, const void *v, const void *o, const float *lse, int B,
                   int H, int L, int D, int mask_kind, int block_size, float sm_scale, int dtype) {
    bool go = false;
    return check_fwd_args<false>(q, k, v, o, lse, B, H, L, D, mask_kind, block_size, sm_scale, dtype, &go);
}

int attn_fwd_fp8v_check(const void *q, const void *k, const void *vt, const void *o, const float *lse,
                        int B, int H, int L, int D, int mask_kind, int block_size, float sm_scale,
                        int dtype) {
    bool go = false;
    return check_fwd_args<true>(q, k, vt, o, lse, B, H, L, D, mask_kind, block_size, sm_scale, dtype, &go);
}

int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int L,
             int D, int mask_kind, int block_size, float sm_scale, int dtype, void *stream) {
    return fwd_common<false>(q, k, v, o, lse, B, H, L, D, mask_kind, block_size, sm_scale, dtype, stream);
}

int attn_fwd_fp8v(const void *q, const void *k, const void *vt, void *o, float *lse, int B, int H, int L,
                  int D, int mask_kind, int block_size, float sm_scale, int dtype, void *stream) {
    return fwd_common<true>(q, k, vt, o, lse, B, H, L, D, mask_kind, block_size, sm_scale, dtype, stream);
}

int attn_last_device_status(int device, int *status, unsigned int *detail) {
    if (!status) return ATTN_ERR_NULL;
    if (device < 0 || device >= kMaxDevices) return ATTN_ERR_ARG;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaSetDevice(device) != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned int word = 0;
    int rc = ATTN_OK;
    {
        std::lock_guard<std::mutex> lk(g_mutex);
        DeviceState &st = g_dev[device];
        if (st.ready) {
            if (cudaDeviceSynchronize() != cudaSuccess ||
                cudaMemcpy(&word, st.status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess ||
                cudaMemset(st.status, 0, sizeof word) != cudaSuccess)
                rc = ATTN_ERR_CUDA;
        }
    }
    cudaSetDevice(prev);
    if (rc != ATTN_OK) return rc;
    *status = static_cast<int>(word & 0xffu);   // 0, ATTN_ERR_TIMEOUT or ATTN_ERR_CUDA
    if (detail) *detail = word;
    return ATTN_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant: the status word lives in a fixed array compiled
// into this library instead of memory cudaMalloc'd per device.

namespace {

constexpr int kNoAllocScratchWords = ATTN_NOALLOC_SCRATCH_BYTES / 4;
static_assert(kNoAllocScratchWords * 4 == ATTN_NOALLOC_SCRATCH_BYTES, "scratch size");

// Word 0: device status of the latest call; the rest is reserved.  Host code
// must not use this name as a device address: it is a host-side stand-in.
static __device__ __align__(256) unsigned int g_noalloc_scratch[kNoAllocScratchWords];

std::mutex g_noalloc_mutex;
DeviceState g_noalloc_dev[kMaxDevices];   // .status = device address of the array

// Set-up, once per device and with that device current: SM count, tensor-map
// encoder, the array's device address, and a cleared array.  No allocation.
int noalloc_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lk(g_mutex);
        int rc = load_encoder();
        if (rc != ATTN_OK) return rc;
    }
    std::lock_guard<std::mutex> lk(g_noalloc_mutex);
    DeviceState &st = g_noalloc_dev[dev];
    if (!st.ready) {
        if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return ATTN_ERR_CUDA;
        if (cudaMemset(ptr, 0, ATTN_NOALLOC_SCRATCH_BYTES) != cudaSuccess) return ATTN_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
        st.status = static_cast<unsigned int *>(ptr);
        st.ready = true;
    }
    *out = &st;
    return ATTN_OK;
}

}  // namespace

extern "C" int attn_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                                int B, int H, int L, int D, int mask_kind, int block_size,
                                float sm_scale, int dtype, void *stream,
                                unsigned int *status_out) {
    bool go = false;
    int rc = check_fwd_args<false>(q, k, v, o, lse, B, H, L, D, mask_kind, block_size, sm_scale, dtype, &go);
    if (rc != ATTN_OK) return rc;
    // scratch this kernel needs: one status word, whatever the problem size
    constexpr size_t kNeeded = sizeof(unsigned int);
    if (kNeeded > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;
    if (!go) {
        if (status_out) *status_out = 0;
        return ATTN_OK;
    }

    DeviceState *st = nullptr;
    rc = noalloc_state(&st);
    if (rc != ATTN_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(st->status, 0, kNeeded, s) != cudaSuccess) return ATTN_ERR_CUDA;

    const Plan pl = make_plan(B, H, L, D);
    FwdParams prm;
    prm.o = o;
    prm.lse = lse;
    prm.status = st->status;
    prm.BH = B * H;
    prm.L = L;
    prm.mask = mask_kind;
    prm.bs = mask_kind == ATTN_MASK_BLOCK_DIAG ? block_size : 0;
    prm.n_qt = pl.n_qt;
    prm.n_kv = pl.n_kv;
    prm.n_units = pl.n_units;
    prm.scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634074);
    prm.inject = 0;
    prm.kv_keep = kv_fits_l2(prm.BH, L, D) ? 1 : 0;
    prm.d_out = D;

    const bool bf16 = dtype == ATTN_BF16;
    const bool bdh = small_blocks(mask_kind, block_size);
    switch (kernel_dim(D)) {
        case 64:
            rc = bdh ? (bf16 ? launch<64, true, true, false, true>(*st, q, k, v, prm, dtype, s)
                             : launch<64, false, true, false, true>(*st, q, k, v, prm, dtype, s))
                     : (bf16 ? launch<64, true, true>(*st, q, k, v, prm, dtype, s)
                             : launch<64, false, true>(*st, q, k, v, prm, dtype, s));
            break;
        case 128:
            rc = bdh ? (bf16 ? launch<128, true, true, false, true>(*st, q, k, v, prm, dtype, s)
                             : launch<128, false, true, false, true>(*st, q, k, v, prm, dtype, s))
                     : (bf16 ? launch<128, true, true>(*st, q, k, v, prm, dtype, s)
                             : launch<128, false, true>(*st, q, k, v, prm, dtype, s));
            break;
        default:
            rc = bf16 ? launch<256, true, false>(*st, q, k, v, prm, dtype, s)
                      : launch<256, false, false>(*st, q, k, v, prm, dtype, s);
            break;
    }
    if (rc != ATTN_OK) return rc;
    if (status_out &&
        cudaMemcpyAsync(status_out, st->status, kNeeded, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}

// ---------------------------------------------------------------------------
// Backward: attn_bwd_workspace_size, attn_bwd, attn_bwd_work.

namespace {

size_t bwd_workspace_bytes(long long BH, int L) {
    const long long n_pad = static_cast<long long>((L + 127) / 128) * 128;
    return static_cast<size_t>(2 * BH * n_pad) * sizeof(float);
}

template <int D, bool BF16, bool DQ>
int launch_bwd(DeviceState &st, const CUtensorMap &f0, const CUtensorMap &f1, const CUtensorMap &r0,
               const CUtensorMap &r1, const CUtensorMap &g0, const CUtensorMap &g1, const attn::BwdParams &prm,
               cudaStream_t stream) {
    using C = attn::BwdCfg<D, DQ>;
    auto kern = attn::attn_bwd_kernel<D, BF16, DQ>;
    {
        std::lock_guard<std::mutex> lk(g_mutex);
        bool &set = st.bwd_attr[D == 64 ? 0 : (D == 128 ? 1 : 2)][BF16 ? 1 : 0][DQ ? 1 : 0];
        if (!set) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
                cudaSuccess)
                return ATTN_ERR_CUDA;
            set = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    // one CTA per (head, fixed tile); DSPLIT: two, one per head-dim half
    cfg.gridDim = dim3(static_cast<unsigned>(prm.BH) * static_cast<unsigned>(prm.n_t) * (C::DSPLIT ? 2u : 1u));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, f0, f1, r0, r1, g0, g1, prm) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// t*: maps with 128-row boxes (fixed tiles, and streamed ones of a whole-tile
// ring); s*: the streamed operands' maps (64-row boxes when the ring holds
// half tiles, D = 256).
template <int D, bool BF16>
int bwd_for_dim(DeviceState &st, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                const CUtensorMap &tg, const CUtensorMap &sq, const CUtensorMap &sk, const CUtensorMap &sv,
                const CUtensorMap &sg, attn::BwdParams prm, void *dq, void *dk, void *dv, cudaStream_t s) {
    // The dQ kernel needs only the prep kernel's vectors, not dK/dV: it runs on a
    // second stream forked after the prep kernel and joined back before return,
    // so its CTAs take the SMs the last wave of dK/dV leaves idle.  The fork/join
    // is held under the library lock, so that concurrent callers cannot
    // interleave the shared events, and is legal inside stream capture.
    std::lock_guard<std::mutex> lk(g_bwd_mutex);
    if (!st.side) {
        if (cudaStreamCreateWithFlags(&st.side, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&st.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&st.join, cudaEventDisableTiming) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    if (cudaEventRecord(st.fork, s) != cudaSuccess || cudaStreamWaitEvent(st.side, st.fork, 0) != cudaSuccess)
        return ATTN_ERR_CUDA;
    // output maps (dK, dV, dQ) for the kernels' staged stores
    const int dt = BF16 ? ATTN_BF16 : ATTN_F16;
    CUtensorMap mdk, mdv, mdq, none;
    std::memset(&none, 0, sizeof(none));
    int rc = encode_store_map(&mdk, dk, prm.BH, prm.L, prm.d_out, dt);
    if (rc == ATTN_OK) rc = encode_store_map(&mdv, dv, prm.BH, prm.L, prm.d_out, dt);
    if (rc == ATTN_OK) rc = encode_store_map(&mdq, dq, prm.BH, prm.L, prm.d_out, dt);
    // dK/dV: fixed K, V; streamed Q, dO
    prm.g0 = dk;
    prm.g1 = dv;
    if (rc == ATTN_OK) rc = launch_bwd<D, BF16, false>(st, tk, tv, sq, sg, mdk, mdv, prm, s);
    // dQ: fixed Q, dO; streamed K, V
    prm.g0 = dq;
    prm.g1 = nullptr;
    if (rc == ATTN_OK) rc = launch_bwd<D, BF16, true>(st, tq, tg, sk, sv, mdq, none, prm, st.side);
    // the caller's stream waits for the dQ kernel (joined even after a failed
    // launch, so that the side stream never stays forked)
    if (cudaEventRecord(st.join, st.side) != cudaSuccess || cudaStreamWaitEvent(s, st.join, 0) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return rc;
}

}  // namespace

extern "C" {

size_t attn_bwd_workspace_size(int B, int H, int L) {
    if (B < 0 || H < 0 || L < 0) return 0;
    return bwd_workspace_bytes(static_cast<long long>(B) * H, L);
}

int attn_bwd_check(const void *q, const void *k, const void *v, const void *o, const void *dout,
                   const float *lse, const void *dq, const void *dk, const void *dv, const void *workspace,
                   size_t workspace_bytes, int B, int H, int L, int D, int mask_kind, int block_size,
                   float sm_scale, int dtype) {
    int rc = validate_shape(B, H, L, D, mask_kind, block_size, dtype);
    if (rc != ATTN_OK) return rc;
    if (!std::isfinite(sm_scale)) return ATTN_ERR_ARG;
    if (static_cast<long long>(B) * H * L == 0) return ATTN_OK;   // empty problem
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace) return ATTN_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
        !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
        return ATTN_ERR_ALIGN;
    if (workspace_bytes < bwd_workspace_bytes(static_cast<long long>(B) * H, L)) return ATTN_ERR_ARG;
    return ATTN_OK;
}

int attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout, const float *lse,
             void *dq, void *dk, void *dv, void *workspace, size_t workspace_bytes, int B, int H, int L, int D,
             int mask_kind, int block_size, float sm_scale, int dtype, void *stream) {
    int rc = attn_bwd_check(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, L, D,
                            mask_kind, block_size, sm_scale, dtype);
    if (rc != ATTN_OK) return rc;
    if (static_cast<long long>(B) * H * L == 0) return ATTN_OK;   // empty problem
    const long long bh = static_cast<long long>(B) * H;

    DeviceState *st = nullptr;
    rc = device_state(&st, nullptr);
    if (rc != ATTN_OK) return rc;

    attn::BwdParams prm = {};
    prm.o = o;
    prm.dout = dout;
    prm.lse = lse;
    prm.status = st->status;
    prm.BH = static_cast<int>(bh);
    prm.L = L;
    prm.mask = mask_kind;
    prm.bs = mask_kind == ATTN_MASK_BLOCK_DIAG ? block_size : 0;
    prm.n_t = (L + 127) / 128;
    prm.n_pad = prm.n_t * 128;
    prm.nlse2 = static_cast<float *>(workspace);
    prm.ndelta = prm.nlse2 + static_cast<size_t>(bh) * prm.n_pad;
    prm.scale = sm_scale;
    prm.scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634074);
    prm.d_out = D;
    prm.inject = g_inject;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool bf16 = dtype == ATTN_BF16;
    // -Di and -lse * log2(e), padded per head
    {
        const long long rows = bh * prm.n_pad;
        long long blocks = (rows + 31) / 32;
        const long long cap = static_cast<long long>(st->sms) * 16;
        if (blocks > cap) blocks = cap;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(blocks));
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = bf16 ? cudaLaunchKernelEx(&cfg, attn::attn_bwd_prep_kernel<true>, prm)
                             : cudaLaunchKernelEx(&cfg, attn::attn_bwd_prep_kernel<false>, prm);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return ATTN_ERR_CUDA;
        }
    }
    CUtensorMap tq, tk, tv, tg;
    rc = encode_map(&tq, q, prm.BH, L, D, dtype);
    if (rc == ATTN_OK) rc = encode_map(&tk, k, prm.BH, L, D, dtype);
    if (rc == ATTN_OK) rc = encode_map(&tv, v, prm.BH, L, D, dtype);
    if (rc == ATTN_OK) rc = encode_map(&tg, dout, prm.BH, L, D, dtype);
    if (rc != ATTN_OK) return rc;
    if (kernel_dim(D) == 64)
        return bf16 ? bwd_for_dim<64, true>(*st, tq, tk, tv, tg, tq, tk, tv, tg, prm, dq, dk, dv, s)
                    : bwd_for_dim<64, false>(*st, tq, tk, tv, tg, tq, tk, tv, tg, prm, dq, dk, dv, s);
    if (kernel_dim(D) == 128)
        return bf16 ? bwd_for_dim<128, true>(*st, tq, tk, tv, tg, tq, tk, tv, tg, prm, dq, dk, dv, s)
                    : bwd_for_dim<128, false>(*st, tq, tk, tv, tg, tq, tk, tv, tg, prm, dq, dk, dv, s);
    // D = 256: the streamed operands travel as 64-row halves
    CUtensorMap sq, sk, sv, sg;
    rc = encode_map(&sq, q, prm.BH, L, D, dtype, 64);
    if (rc == ATTN_OK) rc = encode_map(&sk, k, prm.BH, L, D, dtype, 64);
    if (rc == ATTN_OK) rc = encode_map(&sv, v, prm.BH, L, D, dtype, 64);
    if (rc == ATTN_OK) rc = encode_map(&sg, dout, prm.BH, L, D, dtype, 64);
    if (rc != ATTN_OK) return rc;
    return bf16 ? bwd_for_dim<256, true>(*st, tq, tk, tv, tg, sq, sk, sv, sg, prm, dq, dk, dv, s)
                : bwd_for_dim<256, false>(*st, tq, tk, tv, tg, sq, sk, sv, sg, prm, dq, dk, dv, s);
}

int attn_bwd_work(int B, int H, int L, int D, int mask_kind, int block_size, int dtype, double *flops,
                  double *bytes) {
    int rc = validate_shape(B, H, L, D, mask_kind, block_size, dtype);
    if (rc != ATTN_OK) return rc;
    double f = 0.0;
    rc = attn_fwd_work(B, H, L, D, mask_kind, block_size, dtype, &f, nullptr);
    if (rc != ATTN_OK) return rc;
    // five products of the forward's size (S, dP, dV, dK, dQ); the dQ kernel's
    // second S and dP are not counted
    if (flops) *flops = 2.5 * f;
    // q, k, v, o, dO read and dq, dk, dv written once, lse read once
    if (bytes) *bytes = (8.0 * 2.0 * D + 4.0) * static_cast<double>(B) * H * L;
    return ATTN_OK;
}

}  // extern "C"
