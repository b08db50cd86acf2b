// Fused attention forward for sm_103a (GB300): TMA -> shared memory ->
// tcgen05.mma into tensor memory -> online softmax in registers -> tcgen05.mma
// P.V back into tensor memory -> normalised output.
//
// What is computed (per query row i of head (b,h)):
//   O_i   = sum_{j in A(i)} exp(s_ij - m_i) v_j / l_i,   s_ij = sm_scale q_i.k_j
//   lse_i = m_i + ln l_i
// with A(i) the attended keys of the mask kind (dense / causal j <= i /
// block-diagonal floor(j/bs) == floor(i/bs)).  The key axis is walked tile by
// tile with the online-softmax recurrence of the "Triton-CUDA Attention" page
// (running max m, running denominator l, accumulator rescaled by
// exp2(m_old - m_new)), in base 2 with sm_scale*log2(e) folded into one fma.
//
// Structure of one CTA (one CTA per SM, persistent over work units):
//   * warp "TMA"     : one lane issues cp.async.bulk.tensor loads of Q tiles
//                      into dedicated slots and of K/V tiles into a ring;
//   * warp "MMA"     : one lane issues tcgen05.mma: S = Q K^T (both operands
//                      K-major in shared memory, fp32 accumulator in TMEM) and
//                      O += P V (P read from TMEM, V MN-major in shared memory);
//                      it also owns the TMEM allocation;
//   * softmax groups : 4 warps each, one thread per query row (= TMEM lane);
//                      they read S from TMEM, apply the mask only on tiles
//                      that cross it, run the online softmax, write P (16-bit)
//                      over S in TMEM, rescale O in TMEM when the running max
//                      grew past a threshold, and finally write O / l and lse.
// Work is split into units; a unit is one head and one or two 128-row query
// tiles ("lanes") that share the stream of K/V tiles.  Key tiles that lie
// wholly outside a lane's attended range are never loaded or multiplied for it
// (causal: tiles above the diagonal; block-diagonal: tiles of other blocks);
// only tiles that cross the mask boundary go through the masked path.
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   pair mode (D <= 128): S/P lane 0 at col 0, S/P lane 1 at col 128,
//                         O lane 0 at col 256, O lane 1 at col 256 + D;
//   single mode (D = 256): one query tile, two S/P buffers at cols 0 and 128
//                         (consecutive key tiles alternate), O at col 256.
// P (16-bit, two per column) overwrites the upper BN/2 columns of its S.
//
// Every mbarrier wait is bounded (about one second); on expiry the kernel
// records a timeout in the status word, tells the other roles to stop through
// a shared-memory flag, waits (bounded) for its own copies and MMAs in flight,
// frees its tensor memory and returns.
#pragma once

#include <climits>
#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"

namespace attn {

constexpr int BM = 128;                       // query rows per tile (one per TMEM lane)
constexpr int BN = 128;                       // keys per tile
constexpr float kRescaleLog2 = 8.0f;          // rescale O only if the max grows by > 2^8
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr unsigned kStatusTimeout = 7u;       // == ATTN_ERR_TIMEOUT
constexpr unsigned kStatusTmem = 6u;          // == ATTN_ERR_CUDA: TMEM base not at column 0

enum : int { kMaskDense = 0, kMaskCausal = 1, kMaskBlock = 2 };

struct FwdParams {
    void *o;                 // [BH, L, D] 16-bit
    float *lse;              // [BH, L] or nullptr
    unsigned int *status;    // device status word
    int BH, L, mask, bs;
    int n_qt, n_kv;          // query / key tiles per head
    int n_units;
    float scale_log2;        // sm_scale * log2(e)
    int kv_keep;             // 1: K/V loads ask L2 to keep them (all K/V fit in L2)
    int inject;              // test hook: 1 = the producer issues no copies, so every
                             // consumer's bounded wait runs out (0 in normal use)
    int d_out;               // head dim of Q, K, V and O in memory (<= D of the kernel;
                             // the columns past it load as zeros and are not stored)
};

template <int D, bool PAIR, bool FP8V = false>
struct Cfg {
    static constexpr int NQ = PAIR ? 2 : 1;           // query tiles resident per CTA
    static constexpr int NWG = PAIR ? 2 : 1;          // softmax warpgroups
    static constexpr int CHUNKS = D / 64;             // 128-byte-wide TMA boxes per row
    static constexpr int CHUNK_BYTES = 128 * 128;     // one box: 128 rows x 128 bytes
    static constexpr int TILE_BYTES = 128 * D * 2;    // one Q, K or V tile
    // K/V ring entries: a whole tile, or (D = 256) half a tile along the head
    // dim, so that a deeper ring fits next to the 64 KB Q tile
    static constexpr int EPT = D == 256 ? 2 : 1;                 // entries per tile
    static constexpr int ENTRY_BYTES = TILE_BYTES / EPT;
    static constexpr int ENTRY_CHUNKS = CHUNKS / EPT;
    // (D = 128 pair mode: four entries, leaving room for the staged O rows)
    static constexpr int RING = D == 64 ? 8 : (PAIR ? 4 : 5);
    // SEP: P has columns of its own (D = 64 leaves room), so the next S of a
    // lane can be computed while the softmax still works on the current one.
    // Then a second MMA warp issues the P.V products, so that neither issuer's
    // barrier waits hold back the other's MMAs.
    static constexpr bool SEP = PAIR && D == 64;
    // REGSPLIT (the FP8 P.V variant in the separate-P mode): the copy and MMA
    // warps fill a whole fourth warpgroup (one warp idle) so that registers can
    // move between warpgroups, and the softmax warpgroups hold a whole S row
    // and the row's packed P in registers (measured faster there; the 16-bit
    // separate-P mode measured faster without it).
    static constexpr bool REGSPLIT = SEP && FP8V;
    static constexpr int NUM_WARPS = REGSPLIT ? 12 : 4 * NWG + 2 + (SEP ? 1 : 0);
    static constexpr int THREADS = 32 * NUM_WARPS;
    static constexpr int WARP_TMA = 4 * NWG;
    static constexpr int WARP_MMA = 4 * NWG + 1;
    static constexpr int WARP_PV = 4 * NWG + 2;     // SEP only
    // REGSPLIT register split (per thread): launched with REGS_LAUNCH, the
    // copy/MMA warpgroup drops to REGS_CTRL and the softmax warpgroups rise to
    // REGS_SOFT; the two splits use the same total.
    static constexpr int REGS_LAUNCH = 168, REGS_CTRL = 56, REGS_SOFT = 224;
    static_assert(!REGSPLIT || 4 * NWG * REGS_SOFT + 4 * REGS_CTRL == NUM_WARPS * REGS_LAUNCH,
                  "register split must use exactly the launch pool");
    // ROW_IN_REGS: the softmax holds a whole 128-key S row in registers (one TMEM
    // round trip per tile): the single mode, and the register-split mode.
    static constexpr bool ROW_IN_REGS = !PAIR || REGSPLIT;
    // TMEM columns of S buffer b, of P buffer b and of the O accumulator of lane w.
    // Without SEP, P (16-bit pairs) occupies the upper BN/2 columns of its S.
    __device__ static constexpr uint32_t s_col(int b) { return static_cast<uint32_t>(b) * 128u; }
    __device__ static constexpr uint32_t p_col(int b) {
        return SEP ? 256u + static_cast<uint32_t>(b) * 64u : s_col(b) + BN / 2;
    }
    // FP8 P.V variant: P as e5m2, four keys per column (32 columns a tile), where
    // it overwrites nothing still to be read: the P columns of its own (SEP),
    // over S keys 96..127, which the softmax holds in registers (pair), or the
    // upper half of a whole-row-in-registers S (single).
    __device__ static constexpr uint32_t pf8_col(int b) {
        return SEP ? p_col(b) : (PAIR ? s_col(b) + 96u : s_col(b) + 64u);
    }
    __device__ static constexpr uint32_t o_col(int w) {
        return SEP ? 384u + static_cast<uint32_t>(w) * 64u
                   : 256u + (PAIR ? static_cast<uint32_t>(w) * D : 0u);
    }
    static constexpr uint32_t TMEM_COLS = 512;
    // shared memory (offsets from a 1024-byte aligned base)
    // Q slots: NQB buffers per lane, so the next unit's Q (and the K/V behind it)
    // can load while the current unit runs; slot (lane w, buffer qb) = qb*NQ + w
    static constexpr int NQB = D == 64 ? 2 : 1;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = NQB * NQ * TILE_BYTES;
    // OSTAGE (pair modes): each softmax warp writes its 32 rows of O through a
    // shared slab of its own, 64 columns (128 bytes a row) per TMA store.  A
    // thread storing its own row from registers touches 32 lines per instruction.
    static constexpr bool OSTAGE = PAIR;
    static constexpr int OST_WARP_BYTES = 32 * 64 * 2;
    static constexpr int OFF_OST = OFF_RING + RING * ENTRY_BYTES;
    static constexpr int OFF_BAR = OFF_OST + (OSTAGE ? 4 * NWG * OST_WARP_BYTES : 0);
    // barrier indices
    static constexpr int B_QFULL = 0, B_QEMPTY = 4, B_KVFULL = 8;
    static constexpr int B_KVEMPTY = B_KVFULL + RING;
    static constexpr int B_SFULL = B_KVEMPTY + RING;
    static constexpr int B_PFULL = B_SFULL + 2;
    static constexpr int B_ODONE = B_PFULL + 2;
    static constexpr int B_SFREE = B_ODONE + 2;     // SEP: S buffer read by the softmax
    static constexpr int B_DRAIN = B_SFREE + 2;
    static constexpr int NBAR = B_DRAIN + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // [0]: TMEM base, [1]: abort flag
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;   // slack for 1024-byte alignment
    static_assert(D == 64 || D == 128 || D == 256, "head dim");
    static_assert(PAIR ? (2 * 128 + 2 * D <= 512) : (D == 256), "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(PAIR ? EPT == 1 : true, "pair modes keep whole-tile ring entries");
    static_assert(!OSTAGE || D <= 128, "staged O: pair modes only");
};

// ------------------------------------------------------------ work units

struct Unit {
    int bh;
    int qt[2];     // query tile of each lane, -1 if the lane is idle in this unit
    int lo[2];     // key-tile range [lo, hi) of each lane
    int hi[2];
    int ulo, uhi;  // union of the lanes' ranges
};

// Key tiles a 128-row query tile attends (tiles wholly outside the mask are
// excluded here, so they are never loaded or multiplied).
__device__ __forceinline__ void kv_range(const FwdParams &p, int qt, int &lo, int &hi) {
    if (p.mask == kMaskDense) {
        lo = 0;
        hi = p.n_kv;
    } else if (p.mask == kMaskCausal) {
        lo = 0;
        hi = qt + 1;                          // BM == BN: the diagonal tile is qt
    } else {
        const int q0 = qt * BM;
        const int q1 = min(q0 + BM, p.L);
        const int klo = (q0 / p.bs) * p.bs;
        const int khi = ((q1 - 1) / p.bs + 1) * p.bs;
        lo = klo / BN;
        hi = (khi + BN - 1) / BN;
    }
}

// True if some (row, key) pair of the tile is outside the mask (or past L),
// i.e. the tile needs the element-wise masked path.
__device__ __forceinline__ bool tile_masked(const FwdParams &p, int qt, int j) {
    if (p.mask == kMaskDense) return (j + 1) * BN > p.L;
    if (p.mask == kMaskCausal) return j == qt;
    return (p.bs % BN) != 0;
}

template <bool PAIR>
__device__ __forceinline__ Unit make_unit(const FwdParams &p, int u) {
    Unit U;
    const int per_bh = PAIR ? (p.n_qt + 1) / 2 : p.n_qt;
    int idx;
    if (p.mask == kMaskCausal) {              // heaviest query tiles first
        idx = per_bh - 1 - u / p.BH;
        U.bh = u % p.BH;
    } else {                                  // neighbouring units share a head
        U.bh = u / per_bh;
        idx = u % per_bh;
    }
    if (PAIR) {
        U.qt[0] = 2 * idx;
        U.qt[1] = (2 * idx + 1 < p.n_qt) ? 2 * idx + 1 : -1;
    } else {
        U.qt[0] = idx;
        U.qt[1] = -1;
    }
    U.ulo = INT_MAX;
    U.uhi = INT_MIN;
    for (int w = 0; w < 2; ++w) {
        if (U.qt[w] >= 0) {
            kv_range(p, U.qt[w], U.lo[w], U.hi[w]);
            U.ulo = min(U.ulo, U.lo[w]);
            U.uhi = max(U.uhi, U.hi[w]);
        } else {
            U.lo[w] = U.hi[w] = 0;
        }
    }
    return U;
}

__device__ __forceinline__ bool lane_uses(const Unit &U, int w, int j) {
    return U.qt[w] >= 0 && j >= U.lo[w] && j < U.hi[w];
}

// Unit taken by CTA `cta` of `G` in round r (>= n_units means none).  Causal
// units are sorted heaviest first and dealt in a snake order so that every
// CTA gets a similar total.
__device__ __forceinline__ int unit_of(const FwdParams &p, int cta, int G, int r) {
    if (p.mask == kMaskCausal && (r & 1)) return r * G + (G - 1 - cta);
    return r * G + cta;
}

// ------------------------------------------------------------ bounded waits

struct Ctl {
    volatile int *abort_flag;
    unsigned int *status;
};

__device__ __forceinline__ bool wait_slow_body(uint32_t bar, uint32_t parity, const Ctl &c, unsigned site,
                                               bool honour_abort) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u) {
            if (honour_abort && *c.abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                griddep_wait();
                atomicCAS(c.status, 0u, kStatusTimeout | (site << 8));
                *c.abort_flag = 1;
                return false;
            }
        }
    }
}

// The slow path of a bounded wait as a call (keeps the callers' code small)
// or inlined (INL: a kernel that moves registers between warpgroups cannot make
// calls, which would cross code regions whose register counts differ).
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Ctl &c, unsigned site,
                                       bool honour_abort) {
    return wait_slow_body(bar, parity, c, site, honour_abort);
}

template <bool INL>
__device__ __forceinline__ bool wait_slow_t(uint32_t bar, uint32_t parity, const Ctl &c, unsigned site,
                                            bool honour_abort) {
    if constexpr (INL)
        return wait_slow_body(bar, parity, c, site, honour_abort);
    else
        return wait_slow(bar, parity, c, site, honour_abort);
}

template <bool INL = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl &c, unsigned site) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow_t<INL>(bar, parity, c, site, true);
}

// wait sites (recorded in the status word on a timeout)
enum : unsigned {
    kSiteQEmpty = 1, kSiteKvEmpty = 2, kSiteQFull = 3, kSiteKvFullK = 4, kSiteKvFullV = 5,
    kSitePFull = 6, kSiteSFull = 7, kSiteODone = 8, kSiteDrain = 9, kSiteSFree = 10
};

// Two counters selected by a runtime index without a local-memory array.
struct Count2 {
    uint32_t v0 = 0, v1 = 0;
    __device__ __forceinline__ uint32_t get(int i) const { return i ? v1 : v0; }
    __device__ __forceinline__ void set(int i, uint32_t x) {
        if (i) v1 = x; else v0 = x;
    }
    __device__ __forceinline__ void inc(int i) {
        if (i) ++v1; else ++v0;
    }
};

// ------------------------------------------------------- softmax helpers

// Keys of a 64-key half (first key index `base` in the tile) outside
// [rel_lo, rel_hi) take the value `fill` (excluded from the row extreme).
__device__ __forceinline__ void mask_half(uint32_t (&v)[64], int base, int rel_lo, int rel_hi,
                                          float fill) {
#pragma unroll
    for (int c = 0; c < 64; ++c)
        if (static_cast<unsigned>(base + c - rel_lo) >= static_cast<unsigned>(rel_hi - rel_lo))
            v[c] = __float_as_uint(fill);
}

// max (or min) of N raw scores (N even, N >= 12) with three-input min/max in
// four chains: keys 0..11 seed the chains three at a time, keys 12..N-1 join
// them two at a time -- N/2 operations in all, the fewest three-input ops can do.
template <int N>
__device__ __forceinline__ float row_extreme_n(const uint32_t *v, bool want_max) {
    static_assert(N % 2 == 0 && N >= 12, "row_extreme_n: N even, at least 12");
    float a[4];
    if (want_max) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            a[e] = fmax3(__uint_as_float(v[3 * e]), __uint_as_float(v[3 * e + 1]), __uint_as_float(v[3 * e + 2]));
#pragma unroll
        for (int c = 12; c < N; c += 2)
            a[(c / 2) & 3] = fmax3(a[(c / 2) & 3], __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
        return fmaxf(fmax3(a[0], a[1], a[2]), a[3]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e)
        a[e] = fmin3(__uint_as_float(v[3 * e]), __uint_as_float(v[3 * e + 1]), __uint_as_float(v[3 * e + 2]));
#pragma unroll
    for (int c = 12; c < N; c += 2)
        a[(c / 2) & 3] = fmin3(a[(c / 2) & 3], __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
    return fminf(fmin3(a[0], a[1], a[2]), a[3]);
}

__device__ __forceinline__ float row_extreme64(const uint32_t (&v)[64], bool want_max) {
    return row_extreme_n<64>(v, want_max);
}

__device__ __forceinline__ float row_extreme32(const uint32_t *v, bool want_max) {
    return row_extreme_n<32>(v, want_max);
}

// p = exp2(s * sc - m) for a 64-key half (keys base..base+63 of the tile):
// packed fma, MUFU ex2, packed partial sums into acc[8], rounding to 16-bit
// pairs and one 32-column TMEM store at `dst`.  The packed fp32x2 builtins
// let the compiler keep operand pairs in register pairs.
template <bool BF16, bool MASKED>
__device__ __forceinline__ void exp_half(const uint32_t (&v)[64], int base, int rel_lo, int rel_hi,
                                         float sc, float neg_m, float2 (&acc)[4], uint32_t dst) {
    const float2 sc2 = make_float2(sc, sc);
    const float2 nm2 = make_float2(neg_m, neg_m);
    uint32_t pk[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])),
                                    sc2, nm2);
        float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        if constexpr (MASKED) {
            const unsigned width = static_cast<unsigned>(rel_hi - rel_lo);
            const int c0 = base + 2 * e;
            if (static_cast<unsigned>(c0 - rel_lo) >= width) pp.x = 0.f;
            if (static_cast<unsigned>(c0 + 1 - rel_lo) >= width) pp.y = 0.f;
        }
        acc[e & 3] = __fadd2_rn(acc[e & 3], pp);
        pk[e] = pack2<BF16>(pp.x, pp.y);
    }
    tmem_st32(dst, pk);
}

// p = exp2(s * sc - m) for a 32-key chunk (keys base..base+31 of the tile):
// packed fma, MUFU ex2, packed partial sums into acc[4], rounding to 16-bit
// pairs in pk.  The packed fp32x2 builtins let the compiler keep operand pairs
// in register pairs; the element-wise mask exists only in the masked
// instantiation, which is chosen once per tile.
template <bool BF16, bool MASKED>
__device__ __forceinline__ void exp_pack16(const uint32_t *v, int base, int rel_lo, int rel_hi, float sc,
                                           float neg_m, float2 (&acc)[4], uint32_t (&pk)[16]) {
    const float2 sc2 = make_float2(sc, sc);
    const float2 nm2 = make_float2(neg_m, neg_m);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])),
                                    sc2, nm2);
        float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        if constexpr (MASKED) {
            const unsigned width = static_cast<unsigned>(rel_hi - rel_lo);
            const int c0 = base + 2 * e;
            if (static_cast<unsigned>(c0 - rel_lo) >= width) pp.x = 0.f;
            if (static_cast<unsigned>(c0 + 1 - rel_lo) >= width) pp.y = 0.f;
        }
        acc[e & 3] = __fadd2_rn(acc[e & 3], pp);
        pk[e] = pack2<BF16>(pp.x, pp.y);
    }
}

// The same with P rounded to float8 e5m2 (the FP8 P.V variant): the 32 keys
// four to a word in pk[8].
template <bool MASKED>
__device__ __forceinline__ void exp_pack8q(const uint32_t *v, int base, int rel_lo, int rel_hi, float sc,
                                           float neg_m, float2 (&acc)[4], uint32_t (&pk)[8]) {
    const float2 sc2 = make_float2(sc, sc);
    const float2 nm2 = make_float2(neg_m, neg_m);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        float4 pp;
        const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1])),
                                     sc2, nm2);
        const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3])),
                                     sc2, nm2);
        pp.x = ex2_approx(x0.x);
        pp.y = ex2_approx(x0.y);
        pp.z = ex2_approx(x1.x);
        pp.w = ex2_approx(x1.y);
        if constexpr (MASKED) {
            const unsigned width = static_cast<unsigned>(rel_hi - rel_lo);
            const int c0 = base + 4 * e;
            if (static_cast<unsigned>(c0 - rel_lo) >= width) pp.x = 0.f;
            if (static_cast<unsigned>(c0 + 1 - rel_lo) >= width) pp.y = 0.f;
            if (static_cast<unsigned>(c0 + 2 - rel_lo) >= width) pp.z = 0.f;
            if (static_cast<unsigned>(c0 + 3 - rel_lo) >= width) pp.w = 0.f;
        }
        acc[(2 * e) & 3] = __fadd2_rn(acc[(2 * e) & 3], make_float2(pp.x, pp.y));
        acc[(2 * e + 1) & 3] = __fadd2_rn(acc[(2 * e + 1) & 3], make_float2(pp.z, pp.w));
        pk[e] = pack4_e5m2(pp.x, pp.y, pp.z, pp.w);
    }
}

// exp_pack16 followed by one 16-column TMEM store of the pairs at `dst`.
template <bool BF16, bool MASKED>
__device__ __forceinline__ void exp_chunk(const uint32_t *v, int base, int rel_lo, int rel_hi,
                                          float sc, float neg_m, float2 (&acc)[4], uint32_t dst) {
    uint32_t pk[16];
    exp_pack16<BF16, MASKED>(v, base, rel_lo, rel_hi, sc, neg_m, acc, pk);
    tmem_st16(dst, pk);
}

// exp_pack8q followed by one 8-column TMEM store of the e5m2 words at `dst`.
template <bool MASKED>
__device__ __forceinline__ void exp_chunk8(const uint32_t *v, int base, int rel_lo, int rel_hi,
                                           float sc, float neg_m, float2 (&acc)[4], uint32_t dst) {
    uint32_t pk[8];
    exp_pack8q<MASKED>(v, base, rel_lo, rel_hi, sc, neg_m, acc, pk);
    tmem_st8(dst, pk);
}

// The exponent chunk of keys [base, base+32) with P stored in the format of the
// variant: 16-bit pairs at p16 + base/2, or e5m2 quads at p8 + base/4.
template <bool BF16, bool MASKED, bool FP8V>
__device__ __forceinline__ void exp_chunk_any(const uint32_t *v, int base, int rel_lo, int rel_hi, float sc,
                                              float neg_m, float2 (&acc)[4], uint32_t p16, uint32_t p8) {
    if constexpr (FP8V)
        exp_chunk8<MASKED>(v, base, rel_lo, rel_hi, sc, neg_m, acc, p8 + static_cast<uint32_t>(base) / 4u);
    else
        exp_chunk<BF16, MASKED>(v, base, rel_lo, rel_hi, sc, neg_m, acc, p16 + static_cast<uint32_t>(base) / 2u);
}

// The same for a 64-key half held in one array.
template <bool BF16, bool MASKED, bool FP8V>
__device__ __forceinline__ void exp_half_any(const uint32_t (&v)[64], int base, int rel_lo, int rel_hi,
                                             float sc, float neg_m, float2 (&acc)[4], uint32_t p16,
                                             uint32_t p8) {
    if constexpr (FP8V) {
        exp_chunk8<MASKED>(v, base, rel_lo, rel_hi, sc, neg_m, acc, p8 + static_cast<uint32_t>(base) / 4u);
        exp_chunk8<MASKED>(v + 32, base + 32, rel_lo, rel_hi, sc, neg_m, acc,
                           p8 + static_cast<uint32_t>(base + 32) / 4u);
    } else {
        exp_half<BF16, MASKED>(v, base, rel_lo, rel_hi, sc, neg_m, acc, p16 + static_cast<uint32_t>(base) / 2u);
    }
}

// Unmasked packs of 32 keys for a later store (16-bit pairs, or e5m2 quads).
template <bool BF16>
__device__ __forceinline__ void exp_pack(const uint32_t *v, float sc, float neg_m, float2 (&acc)[4],
                                         uint32_t (&pk)[16]) {
    exp_pack16<BF16, false>(v, 0, 0, 0, sc, neg_m, acc, pk);
}

__device__ __forceinline__ void exp_pack8(const uint32_t *v, float sc, float neg_m, float2 (&acc)[4],
                                          uint32_t (&pk)[8]) {
    exp_pack8q<false>(v, 0, 0, 0, sc, neg_m, acc, pk);
}

// ---------------------------------------------------------------- kernel

// FP8V: the FP8 P.V variant -- tmap_v maps V^T as float8 e5m2 bytes
// ([B*H, D, L], keys innermost), P is rounded to e5m2 and P.V runs as a
// kind::f8f6f4 MMA; the reference max is the exact running max (threshold 0),
// so P is rounded against the same max as the page's recurrence.
// BDH: the block-diagonal instantiation for blocks of at most 64 keys, whose
// masked tiles read and exponentiate only the half of the tile a row attends.
template <int D, bool BF16, bool PAIR, bool FP8V = false, bool BDH = false>
__global__ void __launch_bounds__(Cfg<D, PAIR, FP8V>::THREADS, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_o,
                const FwdParams p) {
    using C = Cfg<D, PAIR, FP8V>;
    constexpr float kThr = FP8V ? 0.f : kRescaleLog2;      // rescale threshold (log2 units)
    // V^T rows per ring entry (FP8V) and the bytes of such an entry
    constexpr int V8_ROWS = D / C::EPT;
    constexpr int V8_BYTES = V8_ROWS * BN;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar0 = s_base + C::OFF_BAR;
    auto bar = [&](int idx) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(idx); };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    const Ctl ctl{reinterpret_cast<volatile int *>(misc + 1), p.status};

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const int cta = blockIdx.x;
    const int rounds_all = (p.n_units + G - 1) / G;

    if (threadIdx.x == 0) {
        for (int q = 0; q < 4; ++q) {
            mbar_init(bar(C::B_QFULL + q), 1);
            mbar_init(bar(C::B_QEMPTY + q), 1);
        }
        for (int s = 0; s < C::RING; ++s) {
            mbar_init(bar(C::B_KVFULL + s), 1);
            mbar_init(bar(C::B_KVEMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(C::B_SFULL + b), 1);
            mbar_init(bar(C::B_PFULL + b), 4);   // one arrival per softmax warp
            mbar_init(bar(C::B_ODONE + b), 1);
            mbar_init(bar(C::B_SFREE + b), 4);   // one arrival per softmax warp
        }
        mbar_init(bar(C::B_DRAIN), C::SEP ? 2 : 1);   // one commit per MMA-issuing warp
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == C::WARP_TMA && lane == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
        if constexpr (C::OSTAGE) tma_prefetch_desc(&tmap_o);
    }
    if (warp == C::WARP_MMA) {
        tmem_alloc(s_base + C::OFF_MISC, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Launched as a programmatic dependent: global memory may be written by the
    // previous kernel of the stream until it completes.  Only the copy warp
    // (before its first load) and the softmax warps (before their first store)
    // touch global memory, and each waits for that completion there, so the
    // roles' first-unit set-up overlaps the previous kernel's tail.  Dependents
    // of this kernel may be scheduled from now on (they wait in the same way).
    griddep_launch_dependents();
    // Allocating all 512 columns can only start at lane 0, column 0, so the TMEM
    // base is the constant 0 (which keeps every TMEM address a compile-time
    // offset).  Anything else is reported and no work is done.
    constexpr uint32_t tmem = 0;
    const bool tmem_ok = misc[0] == 0u;
    if (!tmem_ok && threadIdx.x == 0) {
        griddep_wait();
        atomicCAS(p.status, 0u, kStatusTmem);
    }

    // Waits in every role are polled by all 32 lanes and their outcome made
    // warp-uniform, so warp-collective instructions after them never diverge.
    auto wait_warp = [&](uint32_t bar_addr, uint32_t parity, unsigned site) -> bool {
        const bool r = wait_bar<C::REGSPLIT>(bar_addr, parity, ctl, site);
        return __all_sync(0xffffffffu, r);
    };

    const int rounds = tmem_ok ? rounds_all : 0;

    // MMA issue helpers (called by a whole converged warp; one elected lane issues)
        constexpr uint32_t IDESC_S = idesc_f16_f32acc(BF16, BM, BN, false);
        constexpr uint32_t IDESC_PV = idesc_f16_f32acc(BF16, BM, D, true);
        constexpr uint32_t IDESC_PV8 = idesc_e5m2_f32acc(BM, D);
        const uint32_t q_smem = s_base + C::OFF_Q;
        const uint32_t ring_smem = s_base + C::OFF_RING;
        // Descriptors advance by adding to their 16-byte-unit address field.
        // S = Q K^T: k-step kk covers head-dim columns [16kk, 16kk+16): box kk/4,
        // 32-byte offset (kk%4) inside the 128-byte swizzled row.
        auto issue_s = [&](int qslot, int sbuf, uint32_t kslot) {
            const uint64_t qd = sdesc_sw128(q_smem + qslot * C::TILE_BYTES, 16, 1024);
            const uint64_t kd = sdesc_sw128(ring_smem + kslot * C::ENTRY_BYTES, 16, 1024);
            const uint32_t d_tmem = tmem + C::s_col(sbuf);
#pragma unroll
            for (int c = 0; c < C::CHUNKS; ++c) {   // four k-steps (32 bytes apart) per box
                const uint64_t off = c * (C::CHUNK_BYTES >> 4);
                mma_ss_x4(d_tmem, qd + off, kd + off, 2, 2, IDESC_S, c > 0 ? 1u : 0u);
            }
        };
        // O += P V: k-step kk covers keys [16kk, 16kk+16) = 16 rows of 128 bytes;
        // consecutive 64-column boxes of V are C::CHUNK_BYTES apart (LBO).
        // (then a commit of the issuing lane's MMAs to `done`)
        auto issue_pv = [&](int sbuf, int ocol_idx, uint32_t vslot, bool accumulate, uint32_t done) {
            const uint32_t d_tmem = tmem + C::o_col(ocol_idx);
            if constexpr (FP8V) {
                // V^T rows of 128 keys (128 bytes, K-major); k-step kk covers keys
                // [32kk, 32kk+32): 32 bytes into the swizzled row, 8 P columns
                const uint64_t vd = sdesc_sw128(ring_smem + vslot * C::ENTRY_BYTES, 16, 1024);
                const uint32_t a = tmem + C::pf8_col(sbuf);
                static_assert(BN / 32 == 4, "one batch of four 32-key steps");
                mma_ts_f8_x4(d_tmem, a, a + 8, a + 16, a + 24, vd, 2, IDESC_PV8, accumulate ? 1u : 0u);
                mma_commit(done);
            } else {
                const uint64_t vd = sdesc_sw128(ring_smem + vslot * C::ENTRY_BYTES, C::CHUNK_BYTES, 1024);
                static_assert(BN / 16 == 8, "one batch of eight 16-key steps");
                mma_ts_x8_commit(d_tmem, tmem + C::p_col(sbuf), vd, 128, IDESC_PV, accumulate ? 1u : 0u, done);
            }
        };

    // Roles by warpgroup first: with REGSPLIT the copy/MMA warpgroup gives
    // registers to the softmax warpgroups, each warpgroup executing one
    // setmaxnreg (the instruction is warpgroup-collective), and the two register
    // counts never meet in shared code before the end of the kernel.
    if (warp >= 4 * C::NWG) {
    if constexpr (C::REGSPLIT) regs_dec<C::REGS_CTRL>();
    if (warp == C::WARP_TMA) {
        // ================================================================ TMA producer
        // (the whole warp runs this loop; one elected lane issues each copy)
        {
            uint32_t rc = 0;             // K/V ring position
            uint32_t qpar = 0;           // bit q: parity of the loads into Q slot q
            uint32_t qused = 0;          // bit q: Q slot q has been loaded
            uint32_t nunit = 0;          // units of this CTA so far
            bool ok = p.inject != 1;
            bool dep = false;            // the previous kernel has completed
            auto dep_wait = [&]() {
                if (!dep) {
                    griddep_wait();
                    dep = true;
                }
            };
            for (int r = 0; r < rounds && ok; ++r) {
                const int u = unit_of(p, cta, G, r);
                if (u >= p.n_units) continue;
                const Unit U = make_unit<PAIR>(p, u);
                const int qb = C::NQB == 2 ? static_cast<int>(nunit & 1u) : 0;
                ++nunit;
#pragma unroll
                for (int w = 0; w < C::NQ; ++w) {
                    if (!ok || U.qt[w] < 0) continue;
                    const int q = qb * C::NQ + w;
                    ok = wait_warp(bar(C::B_QEMPTY + q), ((qpar >> q) & 1u) ^ 1u, kSiteQEmpty);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(C::B_QFULL + q), C::TILE_BYTES);
                    dep_wait();
                    const uint32_t dst = s_base + C::OFF_Q + q * C::TILE_BYTES;
                    for (int c = 0; c < C::CHUNKS; ++c)
                        tma_load_3d(dst + c * C::CHUNK_BYTES, &tmap_q, c * 64, U.qt[w] * BM, U.bh,
                                    bar(C::B_QFULL + q));
                    qpar ^= 1u << q;
                    qused |= 1u << q;
                }
                // one K or V tile of key tile j as EPT ring entries
                auto load_kv = [&](int kind, int j) {
#pragma unroll
                    for (int e = 0; e < C::EPT; ++e) {
                        if (!ok) continue;
                        const uint32_t slot = rc % C::RING;
                        ok = wait_warp(bar(C::B_KVEMPTY + slot), ((rc / C::RING) & 1u) ^ 1u,
                                       kSiteKvEmpty);
                        if (!ok) break;
                        dep_wait();
                        const uint32_t dst = s_base + C::OFF_RING + slot * C::ENTRY_BYTES;
                        if (FP8V && kind == 1) {
                            // V^T: one box of 128 keys (128 bytes) x V8_ROWS head-dim rows
                            mbar_arrive_expect_tx(bar(C::B_KVFULL + slot), V8_BYTES);
                            if (p.kv_keep)
                                tma_load_3d_keep(dst, &tmap_v, j * BN, e * V8_ROWS, U.bh,
                                                 bar(C::B_KVFULL + slot));
                            else
                                tma_load_3d(dst, &tmap_v, j * BN, e * V8_ROWS, U.bh, bar(C::B_KVFULL + slot));
                            ++rc;
                            continue;
                        }
                        mbar_arrive_expect_tx(bar(C::B_KVFULL + slot), C::ENTRY_BYTES);
                        const CUtensorMap *m = kind == 0 ? &tmap_k : &tmap_v;
                        for (int c = 0; c < C::ENTRY_CHUNKS; ++c) {
                            if (p.kv_keep)
                                tma_load_3d_keep(dst + c * C::CHUNK_BYTES, m,
                                                 (e * C::ENTRY_CHUNKS + c) * 64, j * BN, U.bh,
                                                 bar(C::B_KVFULL + slot));
                            else
                                tma_load_3d(dst + c * C::CHUNK_BYTES, m, (e * C::ENTRY_CHUNKS + c) * 64,
                                            j * BN, U.bh, bar(C::B_KVFULL + slot));
                        }
                        ++rc;
                    }
                };
                if constexpr (PAIR) {
                    // per key tile: K, then V.  In the CTA's first unit of a grid
                    // with more units than CTAs, the rest of the ring waits until the
                    // first K has landed: every CTA starts at once, and the first S
                    // should not queue behind the whole grid's ring fill.
                    bool first = nunit == 1 && p.n_units > G;
                    for (int j = U.ulo; j < U.uhi && ok; ++j) {
                        if (!lane_uses(U, 0, j) && !lane_uses(U, 1, j)) continue;
                        const uint32_t kpos = rc;
                        load_kv(0, j);
                        if (first && ok) {
                            ok = wait_warp(bar(C::B_KVFULL + kpos % C::RING), (kpos / C::RING) & 1u, kSiteKvFullK);
                            first = false;
                        }
                        load_kv(1, j);
                    }
                } else {
                    // K runs one tile ahead of V: K(0), then K(t+1), V(t) for each t, so
                    // the next S never waits for the ring space of the V in use
                    const int n = U.hi[0] - U.lo[0];
                    if (n > 0) load_kv(0, U.lo[0]);
                    for (int t = 0; t < n && ok; ++t) {
                        if (t + 1 < n) load_kv(0, U.lo[0] + t + 1);
                        load_kv(1, U.lo[0] + t);
                    }
                }
            }
            if (*ctl.abort_flag) {
                // Stopping early: let the copies already issued land before the
                // CTA's shared memory goes away.
                const uint32_t first = rc > static_cast<uint32_t>(C::RING) ? rc - C::RING : 0u;
                for (uint32_t i = first; i < rc; ++i)
                    wait_slow_t<C::REGSPLIT>(bar(C::B_KVFULL + i % C::RING), (i / C::RING) & 1u, ctl,
                                             kSiteDrain, false);
                for (int q = 0; q < 4; ++q)
                    if ((qused >> q) & 1u)   // the latest load of slot q has parity !bit
                        wait_slow_t<C::REGSPLIT>(bar(C::B_QFULL + q), ((qpar >> q) & 1u) ^ 1u, ctl,
                                                 kSiteDrain, false);
            }
        }
        __syncwarp();
    } else if (warp == C::WARP_MMA) {
        // ================================================================ MMA issuer
        // (the whole warp runs this loop; one elected lane -- always the same
        // one, so its commits cover its MMAs -- issues each tcgen05 instruction)
        {
            uint32_t rc = 0;
            uint32_t qpar = 0;           // bit q: parity of the Q-full waits of slot q
            uint32_t nunit = 0;
            uint32_t pn[2] = {0, 0};     // P-ready waits per S buffer
            uint32_t sfn[2] = {0, 0};    // SEP: S issues per lane (S-free waits)
            bool ok = true;
            for (int r = 0; r < rounds && ok; ++r) {
                const int u = unit_of(p, cta, G, r);
                if (u >= p.n_units) continue;
                const Unit U = make_unit<PAIR>(p, u);
                const int qb = C::NQB == 2 ? static_cast<int>(nunit & 1u) : 0;
                ++nunit;
#pragma unroll
                for (int w = 0; w < C::NQ; ++w) {
                    if (!ok || U.qt[w] < 0) continue;
                    ok = wait_warp(bar(C::B_QFULL + qb * C::NQ + w), (qpar >> (qb * C::NQ + w)) & 1u, kSiteQFull);
                    qpar ^= 1u << (qb * C::NQ + w);
                }
                if (!ok) break;
                tc_fence_after();
                if constexpr (C::SEP) {
                    // Per key tile: S(t+1) of each lane as soon as its softmax has
                    // read S(t); the P.V products are the other MMA warp's.
                    for (int j = U.ulo; j < U.uhi && ok; ++j) {
                        const bool use0 = lane_uses(U, 0, j), use1 = lane_uses(U, 1, j);
                        if (!use0 && !use1) continue;
                        const uint32_t kpos = rc;
                        rc += 2;                                        // K and V entries
                        const uint32_t kslot = kpos % C::RING;
                        ok = wait_warp(bar(C::B_KVFULL + kslot), (kpos / C::RING) & 1u,
                                       kSiteKvFullK);
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int w = 0; w < 2; ++w) {
                            if (!ok || !(w == 0 ? use0 : use1)) continue;
                            ok = wait_warp(bar(C::B_SFREE + w), (sfn[w] & 1u) ^ 1u, kSiteSFree);
                            if (!ok) break;
                            ++sfn[w];
                            tc_fence_after();
                            issue_s(qb * C::NQ + w, w, kslot);
                            mma_commit(bar(C::B_SFULL + w));
                            if (j == U.hi[w] - 1) mma_commit(bar(C::B_QEMPTY + qb * C::NQ + w));
                        }
                        if (!ok) break;
                        mma_commit(bar(C::B_KVEMPTY + kslot));
                    }
                } else if constexpr (PAIR) {
                    int pend_j[2] = {-1, -1};
                    uint32_t pend_v[2] = {0, 0};
                    int npv[2] = {0, 0};
                    auto flush_pv = [&](int w) -> bool {
                        if (!wait_warp(bar(C::B_PFULL + w), pn[w] & 1u, kSitePFull)) return false;
                        ++pn[w];
                        const uint32_t vslot = pend_v[w] % C::RING;
                        if (!wait_warp(bar(C::B_KVFULL + vslot), (pend_v[w] / C::RING) & 1u,
                                       kSiteKvFullV))
                            return false;
                        tc_fence_after();
                        issue_pv(w, w, vslot, npv[w] > 0, bar(C::B_ODONE + w));
                        ++npv[w];
                        const bool other_needs = pend_j[1 - w] == pend_j[w];
                        pend_j[w] = -1;
                        if (!other_needs) mma_commit(bar(C::B_KVEMPTY + vslot));
                        return true;
                    };
                    for (int j = U.ulo; j < U.uhi && ok; ++j) {
                        const bool use0 = lane_uses(U, 0, j), use1 = lane_uses(U, 1, j);
                        if (!use0 && !use1) continue;
                        const uint32_t kpos = rc, vpos = rc + C::EPT;   // EPT = 1 here
                        rc += 2 * C::EPT;
                        const uint32_t kslot = kpos % C::RING;
                        ok = wait_warp(bar(C::B_KVFULL + kslot), (kpos / C::RING) & 1u,
                                       kSiteKvFullK);
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int w = 0; w < 2; ++w) {
                            if (!ok || !(w == 0 ? use0 : use1)) continue;
                            if (pend_j[w] >= 0) ok = flush_pv(w);
                            if (!ok) break;
                            issue_s(qb * C::NQ + w, w, kslot);
                            mma_commit(bar(C::B_SFULL + w));
                            if (j == U.hi[w] - 1) mma_commit(bar(C::B_QEMPTY + qb * C::NQ + w));
                            pend_j[w] = j;
                            pend_v[w] = vpos;
                        }
                        if (ok) mma_commit(bar(C::B_KVEMPTY + kslot));
                    }
#pragma unroll
                    for (int w = 0; w < 2; ++w)
                        if (ok && pend_j[w] >= 0) ok = flush_pv(w);
                } else {
                    // One query tile, S buffers alternate: S(0), S(1), PV(0), S(2), PV(1), ...
                    // A tile's K and V each come as EPT ring entries (head-dim parts):
                    // S takes the k-steps of each K entry in turn; P.V is split along
                    // N into one MMA chain per V entry.
                    constexpr int KS_PER_ENTRY = 4 * C::ENTRY_CHUNKS;          // k-steps
                    constexpr int NV = D / C::EPT;                             // N per part
                    constexpr uint32_t IDESC_PVE = idesc_f16_f32acc(BF16, BM, NV, true);
                    const int n = U.hi[0] - U.lo[0];
                    const uint32_t base = rc;
                    rc += 2u * C::EPT * static_cast<uint32_t>(n);
                    // ring positions in the order the copies are issued: K(0), then
                    // K(t+1), V(t) for each t
                    auto pos_k = [&](int t) -> uint32_t {
                        return base + static_cast<uint32_t>(C::EPT * (t == 0 ? 0 : 2 * t - 1));
                    };
                    auto pos_v = [&](int t) -> uint32_t {
                        return base + static_cast<uint32_t>(C::EPT * (t + 1 < n ? 2 * t + 2 : 2 * t + 1));
                    };
                    auto do_s = [&](int t) -> bool {
                        const uint32_t kpos = pos_k(t);
                        const uint64_t qd = sdesc_sw128(q_smem + qb * C::NQ * C::TILE_BYTES, 16, 1024);
                        const uint32_t d_tmem = tmem + C::s_col(t & 1);
#pragma unroll
                        for (int e = 0; e < C::EPT; ++e) {
                            const uint32_t kslot = (kpos + e) % C::RING;
                            if (!wait_warp(bar(C::B_KVFULL + kslot), ((kpos + e) / C::RING) & 1u,
                                           kSiteKvFullK))
                                return false;
                            tc_fence_after();
                            const uint64_t kd = sdesc_sw128(ring_smem + kslot * C::ENTRY_BYTES, 16, 1024);
#pragma unroll
                            for (int j = 0; j < C::ENTRY_CHUNKS; ++j) {   // four k-steps per box
                                const int cq = e * C::ENTRY_CHUNKS + j;      // box of Q
                                mma_ss_x4(d_tmem, qd + cq * (C::CHUNK_BYTES >> 4), kd + j * (C::CHUNK_BYTES >> 4), 2,
                                          2, IDESC_S, cq > 0 ? 1u : 0u);
                            }
                            // this K entry is free once its k-steps are done
                            mma_commit(bar(C::B_KVEMPTY + kslot));
                        }
                        mma_commit(bar(C::B_SFULL + (t & 1)));
                        if (t == n - 1) mma_commit(bar(C::B_QEMPTY + qb * C::NQ));
                        return true;
                    };
                    ok = do_s(0);
                    for (int t = 0; t < n && ok; ++t) {
                        if (t + 1 < n) ok = do_s(t + 1);
                        if (!ok) break;
                        const int b = t & 1;
                        ok = wait_warp(bar(C::B_PFULL + b), pn[b] & 1u, kSitePFull);
                        if (!ok) break;
                        ++pn[b];
                        const uint32_t vpos = pos_v(t);
#pragma unroll
                        for (int e = 0; e < C::EPT; ++e) {
                            if (!ok) continue;
                            const uint32_t vslot = (vpos + e) % C::RING;
                            ok = wait_warp(bar(C::B_KVFULL + vslot), ((vpos + e) / C::RING) & 1u,
                                           kSiteKvFullV);
                            if (!ok) break;
                            tc_fence_after();
                            const uint32_t d_tmem = tmem + C::o_col(0) + e * NV;
                            if constexpr (FP8V) {
                                constexpr uint32_t IDESC_PVE8 = idesc_e5m2_f32acc(BM, NV);
                                const uint64_t vd = sdesc_sw128(ring_smem + vslot * C::ENTRY_BYTES, 16, 1024);
                                const uint32_t a = tmem + C::pf8_col(b);
                                mma_ts_f8_x4(d_tmem, a, a + 8, a + 16, a + 24, vd, 2, IDESC_PVE8, t > 0 ? 1u : 0u);
                            } else {
                                const uint64_t vd = sdesc_sw128(ring_smem + vslot * C::ENTRY_BYTES,
                                                                C::CHUNK_BYTES, 1024);
                                const uint32_t a_tmem = tmem + C::p_col(b);
#pragma unroll
                                for (int h = 0; h < BN / 64; ++h) {   // four 16-key steps per batch
                                    const uint32_t a = a_tmem + 32 * h;
                                    mma_ts_x4(d_tmem, a, a + 8, a + 16, a + 24, vd + static_cast<uint64_t>(h * 512),
                                              128, IDESC_PVE, (t > 0 || h > 0) ? 1u : 0u);
                                }
                            }
                            // this V entry is free once its part of P.V is done
                            mma_commit(bar(C::B_KVEMPTY + vslot));
                        }
                        if (!ok) break;
                        mma_commit(bar(C::B_ODONE + b));
                    }
                }
            }
            // Every MMA (and the barrier arrivals its commits make) must be done
            // before the CTA frees its tensor memory and exits.
            mma_commit(bar(C::B_DRAIN));
            wait_slow_t<C::REGSPLIT>(bar(C::B_DRAIN), 0, ctl, kSiteDrain, false);
        }
        __syncwarp();
    } else if (C::SEP && warp == C::WARP_PV) {
        // ================================================================ P.V issuer
        // (separate-P pair mode; whole warp converged, one elected lane issues):
        // O_w += P_w V for each lane as soon as its P arrives, lane 0 first.
        {
            uint32_t rc = 0;
            uint32_t pn[2] = {0, 0};     // P-ready waits per lane
            bool ok = true;
            for (int r = 0; r < rounds && ok; ++r) {
                const int u = unit_of(p, cta, G, r);
                if (u >= p.n_units) continue;
                const Unit U = make_unit<PAIR>(p, u);
                int npv[2] = {0, 0};
                for (int j = U.ulo; j < U.uhi && ok; ++j) {
                    const bool use0 = lane_uses(U, 0, j), use1 = lane_uses(U, 1, j);
                    if (!use0 && !use1) continue;
                    const uint32_t vpos = rc + 1;
                    rc += 2;                                            // K and V entries
                    const uint32_t vslot = vpos % C::RING;
                    // V lands long before the first P of the tile: wait for it first,
                    // so that only the P-ready wait stands between P and its MMAs
                    ok = wait_warp(bar(C::B_KVFULL + vslot), (vpos / C::RING) & 1u, kSiteKvFullV);
                    if (!ok) break;
#pragma unroll
                    for (int w = 0; w < 2; ++w) {
                        if (!ok || !(w == 0 ? use0 : use1)) continue;
                        ok = wait_warp(bar(C::B_PFULL + w), pn[w] & 1u, kSitePFull);
                        if (!ok) break;
                        ++pn[w];
                        tc_fence_after();
                        issue_pv(w, w, vslot, npv[w] > 0, bar(C::B_ODONE + w));
                        ++npv[w];
                    }
                    if (!ok) break;
                    mma_commit(bar(C::B_KVEMPTY + vslot));
                }
            }
            mma_commit(bar(C::B_DRAIN));
            wait_slow_t<C::REGSPLIT>(bar(C::B_DRAIN), 0, ctl, kSiteDrain, false);
        }
        __syncwarp();
    }  // (REGSPLIT: the fourth warp of the copy/MMA warpgroup has no role)
    } else {
        // ================================================================ softmax groups
        if constexpr (C::REGSPLIT) regs_inc<C::REGS_SOFT>();
        const int wg = warp >> 2;                       // lane (query tile slot) of this group
        const int wq = warp & 3;                        // TMEM lane quarter of this warp
        const int row = wq * 32 + lane;                 // query row inside the tile
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const float sc = p.scale_log2;
        const float fill = sc >= 0.f ? -INFINITY : INFINITY;
        Count2 sn, made, seen;        // per S buffer: S-ready waits, P tiles handed
                                      // to the MMA warp, P.V completions confirmed
        bool ok = true;
        bool dep = false;             // the previous kernel has completed

        auto wait_pv = [&](int b) -> bool {
            if (seen.get(b) < made.get(b)) {
                if (!wait_warp(bar(C::B_ODONE + b), (made.get(b) - 1) & 1u, kSiteODone)) return false;
                seen.set(b, made.get(b));
            }
            return true;
        };

        for (int r = 0; r < rounds && ok; ++r) {
            const int u = unit_of(p, cta, G, r);
            if (u >= p.n_units) continue;
            const Unit U = make_unit<PAIR>(p, u);
            const int qt = wg ? U.qt[1] : U.qt[0];
            const int j_lo = wg ? U.lo[1] : U.lo[0];
            const int j_hi = wg ? U.hi[1] : U.hi[0];
            if (qt < 0) continue;
            const int i = qt * BM + row;                // query row in the head
            const bool row_valid = i < p.L;
            // attended keys of row i: [klo, khi)
            int klo, khi;
            if (p.mask == kMaskDense) {
                klo = 0;
                khi = p.L;
            } else if (p.mask == kMaskCausal) {
                klo = 0;
                khi = i + 1;
            } else {
                klo = (i / p.bs) * p.bs;
                khi = klo + p.bs;
            }
            float m_ref = -INFINITY;                    // running max (log2 units, may lag)
            float l = 0.f;                              // running denominator
            for (int t = 0; t < j_hi - j_lo && ok; ++t) {
                const int j = j_lo + t;
                const int b = PAIR ? wg : (t & 1);
                ok = wait_warp(bar(C::B_SFULL + b), sn.get(b) & 1u, kSiteSFull);
                if (!ok) break;
                sn.inc(b);
                tc_fence_after();
                const uint32_t s_addr = tmem + lane_off + C::s_col(b);
                const uint32_t p_addr = tmem + lane_off + C::p_col(b);
                const uint32_t p8_addr = tmem + lane_off + C::pf8_col(b);   // FP8V
                const bool masked = tile_masked(p, qt, j);
                const int rel_lo = klo - j * BN, rel_hi = khi - j * BN;
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
                float alpha = 1.f;
                bool rescale = false;
                float neg_m = 0.f;
                if constexpr (C::ROW_IN_REGS) {
                    // Pass 1: the whole S row into registers (one TMEM round trip), then
                    // its extreme (max for sm_scale >= 0, else min).
                    uint32_t sv[BN];
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c)
                        tmem_ld32(s_addr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c));
                    tmem_wait_ld();
                    if constexpr (C::SEP) {
                        // S is read: the MMA warp may overwrite it with the next tile
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(C::B_SFREE + wg));
                    }
                    if (masked) {
                        mask_half(*reinterpret_cast<uint32_t(*)[64]>(sv), 0, rel_lo, rel_hi, fill);
                        mask_half(*reinterpret_cast<uint32_t(*)[64]>(sv + 64), 64, rel_lo, rel_hi, fill);
                    }
                    const float ext = row_extreme_n<BN>(sv, sc >= 0.f);
                    const float m_tile = isinf(ext) ? -INFINITY : ext * sc;
                    if (t == 0) {
                        m_ref = m_tile;
                    } else if (m_tile > m_ref + kThr) {
                        alpha = ex2_approx(m_ref - m_tile);
                        m_ref = m_tile;
                        rescale = true;
                    }
                    neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
                    if constexpr (C::SEP) {
                        // The whole row's P into registers first: the P columns (and O)
                        // of this lane are still read (written) by the previous tile's
                        // P.V until it completes, which is waited for only before the
                        // stores.  (FP8V: e5m2 words, four keys each.)
                        constexpr int PW = FP8V ? 8 : 16;      // words per 32 keys
                        uint32_t pk[BN / 32][PW];
                        if (masked) {
#pragma unroll
                            for (int c = 0; c < BN / 32; ++c) {
                                if constexpr (FP8V)
                                    exp_pack8q<true>(sv + 32 * c, 32 * c, rel_lo, rel_hi, sc, neg_m, acc, pk[c]);
                                else
                                    exp_pack16<BF16, true>(sv + 32 * c, 32 * c, rel_lo, rel_hi, sc, neg_m, acc, pk[c]);
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < BN / 32; ++c) {
                                if constexpr (FP8V)
                                    exp_pack8q<false>(sv + 32 * c, 32 * c, rel_lo, rel_hi, sc, neg_m, acc, pk[c]);
                                else
                                    exp_pack16<BF16, false>(sv + 32 * c, 32 * c, rel_lo, rel_hi, sc, neg_m, acc, pk[c]);
                            }
                        }
                        if (t > 0) {
                            ok = wait_pv(wg);
                            if (!ok) break;
                            tc_fence_after();
                        }
#pragma unroll
                        for (int c = 0; c < BN / 32; ++c) {
                            if constexpr (FP8V)
                                tmem_st8(p8_addr + 8 * c, pk[c]);
                            else
                                tmem_st16(p_addr + 16 * c, pk[c]);
                        }
                    } else {
                        // Pass 2: P = exp2(s*scale - m) in 32-key chunks, rounded and
                        // written over the upper half of this S (whose values are
                        // already in registers); the previous tile's P.V used the other
                        // S buffer.
                        if (masked) {
#pragma unroll
                            for (int c = 0; c < BN / 32; ++c)
                                exp_chunk_any<BF16, true, FP8V>(sv + 32 * c, 32 * c, rel_lo, rel_hi, sc, neg_m, acc, p_addr, p8_addr);
                        } else {
#pragma unroll
                            for (int c = 0; c < BN / 32; ++c)
                                exp_chunk_any<BF16, false, FP8V>(sv + 32 * c, 32 * c, rel_lo, rel_hi, sc, neg_m, acc, p_addr, p8_addr);
                        }
                    }
                } else {
                    bool done = false;
                    if constexpr (PAIR && !C::SEP) {
                        // One pass against the running reference max with P over the
                        // upper half of S: the whole row is checked against the
                        // reference before the first P store, so a tile that climbs more
                        // than the rescale threshold above it falls to the two-pass path
                        // below with S intact.  Keys 64..127 stay in registers (their
                        // columns take P); keys 0..63 are read twice.
                        if (t > 0 && !masked) {
                            uint32_t hi[64], lo[32];
                            tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(hi));
                            tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(hi + 32));
                            tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(lo));
                            tmem_wait_ld();
                            const bool want_max = sc >= 0.f;
                            float ext = row_extreme64(hi, want_max);
                            const float e0 = row_extreme32(lo, want_max);
                            ext = want_max ? fmaxf(ext, e0) : fminf(ext, e0);
                            tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(lo));
                            tmem_wait_ld();
                            const float e1 = row_extreme32(lo, want_max);
                            ext = want_max ? fmaxf(ext, e1) : fminf(ext, e1);
                            const bool fits = m_ref != -INFINITY && ext * sc <= m_ref + kThr;
                            if (__all_sync(0xffffffffu, fits)) {
                                neg_m = -m_ref;
                                tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(lo));
                                exp_chunk_any<BF16, false, FP8V>(hi, 64, rel_lo, rel_hi, sc, neg_m, acc, p_addr, p8_addr);
                                exp_chunk_any<BF16, false, FP8V>(hi + 32, 96, rel_lo, rel_hi, sc, neg_m, acc, p_addr, p8_addr);
                                tmem_wait_ld();
                                tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(hi));
                                exp_chunk_any<BF16, false, FP8V>(lo, 0, rel_lo, rel_hi, sc, neg_m, acc, p_addr, p8_addr);
                                tmem_wait_ld();
                                exp_chunk_any<BF16, false, FP8V>(hi, 32, rel_lo, rel_hi, sc, neg_m, acc, p_addr, p8_addr);
                                done = true;
                            }
                        }
                    }
                    if constexpr (C::SEP) {
                        // One pass against the running reference max.  S stays in TMEM
                        // until this tile's S-free arrival (P has columns of its own),
                        // so a tile whose scores climb more than the rescale threshold
                        // above the reference is simply redone by the two-pass path
                        // below; such tiles are rare once a row has seen a few keys.
                        if (t > 0 && !masked) {
                            uint32_t sv[64];
                            tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(sv));
                            tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
                            tmem_wait_ld();
                            const float lim = m_ref + kThr;
                            bool fits = m_ref != -INFINITY &&
                                        row_extreme64(sv, sc >= 0.f) * sc <= lim;
                            if (__all_sync(0xffffffffu, fits)) {
                                neg_m = -m_ref;
                                // keys 0..63 from registers while keys 64..127 load; their
                                // P waits in registers while the previous tile's P.V still
                                // reads the P columns
                                // (FP8V: e5m2 words, four keys each, in 8-column stores)
                                uint32_t pk0[FP8V ? 8 : 16], pk1[FP8V ? 8 : 16];
                                if constexpr (FP8V) exp_pack8(sv, sc, neg_m, acc, pk0);
                                else exp_pack<BF16>(sv, sc, neg_m, acc, pk0);
                                tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(sv));
                                if constexpr (FP8V) exp_pack8(sv + 32, sc, neg_m, acc, pk1);
                                else exp_pack<BF16>(sv + 32, sc, neg_m, acc, pk1);
                                // No TMEM load is left in flight across the wait below: its
                                // slow path is a call, around which live registers may be
                                // saved and restored, and the destination registers of a
                                // load are undefined until tcgen05.wait::ld.
                                tmem_wait_ld();
                                ok = wait_pv(wg);
                                if (!ok) break;
                                tc_fence_after();
                                tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
                                if constexpr (FP8V) {
                                    tmem_st8(p8_addr, pk0);
                                    tmem_st8(p8_addr + 8, pk1);
                                } else {
                                    tmem_st16(p_addr, pk0);
                                    tmem_st16(p_addr + 16, pk1);
                                }
                                tmem_wait_ld();
                                fits = row_extreme64(sv, sc >= 0.f) * sc <= lim;
                                if (__all_sync(0xffffffffu, fits)) {
                                    // last read of this S: the MMA warp may overwrite it now
                                    tc_fence_before();
                                    __syncwarp();
                                    if (lane == 0) mbar_arrive(bar(C::B_SFREE + wg));
                                    exp_chunk_any<BF16, false, FP8V>(sv, 64, rel_lo, rel_hi, sc, neg_m, acc, p_addr, p8_addr);
                                    exp_chunk_any<BF16, false, FP8V>(sv + 32, 96, rel_lo, rel_hi, sc, neg_m, acc, p_addr, p8_addr);
                                    done = true;
                                } else {
                                    // redo the whole tile: forget the first half's sums and
                                    // let its P stores land before they are overwritten
                                    tmem_wait_st();
#pragma unroll
                                    for (int e = 0; e < 4; ++e) acc[e] = make_float2(0.f, 0.f);
                                }
                            }
                        }
                    }
                    if (!done) {
                        // Pass 1: row extreme (max for sm_scale >= 0, else min) over the
                        // two 64-key halves; the upper half stays in registers.
                        // one_half: block-diagonal with blocks of at most 64 keys, where
                        // a row's keys lie in one 64-key half of the tile, the same half
                        // for every row of the warp (blocks never straddle key 64 and a
                        // warp's 32 rows share one 64-row block): only that half (hv) is
                        // read and exponentiated, and the other half's P is zero.
                        const bool one_half = BDH && masked && p.mask == kMaskBlock && p.bs <= 64;
                        const int hv = one_half && rel_lo < 64 ? 0 : 1;   // the half held in hi
                        uint32_t hi[64];
                        float ext;
                        if (one_half) {
                            tmem_ld32(s_addr + 64 * hv, *reinterpret_cast<uint32_t(*)[32]>(hi));
                            tmem_ld32(s_addr + 64 * hv + 32, *reinterpret_cast<uint32_t(*)[32]>(hi + 32));
                            tmem_wait_ld();
                            if constexpr (C::SEP) {
                                // last read of this S: the MMA warp may overwrite it now
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0) mbar_arrive(bar(C::B_SFREE + wg));
                            }
                            mask_half(hi, 64 * hv, rel_lo, rel_hi, fill);
                            ext = row_extreme64(hi, sc >= 0.f);
                        } else {
                        {
                            uint32_t lo[64];
                            tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(lo));
                            tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(lo + 32));
                            tmem_wait_ld();
                            // the upper half loads while the lower half is reduced
                            tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(hi));
                            tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(hi + 32));
                            if (masked) mask_half(lo, 0, rel_lo, rel_hi, fill);
                            ext = row_extreme64(lo, sc >= 0.f);
                        }
                        tmem_wait_ld();
                        if (masked) mask_half(hi, 64, rel_lo, rel_hi, fill);
                        {
                            const float e2 = row_extreme64(hi, sc >= 0.f);
                            ext = sc >= 0.f ? fmaxf(ext, e2) : fminf(ext, e2);
                        }
                        }
                        const float m_tile = isinf(ext) ? -INFINITY : ext * sc;
                        if (t == 0) {
                            m_ref = m_tile;
                        } else if (m_tile > m_ref + kThr) {
                            alpha = ex2_approx(m_ref - m_tile);
                            m_ref = m_tile;
                            rescale = true;
                        }
                        neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
                        if constexpr (C::SEP) {
                            // P and O of this lane are still read/written by the previous
                            // tile's P.V until it completes.
                            if (t > 0) {
                                ok = wait_pv(wg);
                                if (!ok) break;
                                tc_fence_after();
                            }
                        }

                        // Pass 2: P = exp2(s*scale - m) written as 16-bit pairs into the
                        // upper half of the S columns: the upper 64 keys first (their S
                        // columns are already in registers), then the lower 64 keys,
                        // reloaded (their P columns overwrite S columns 64..95, consumed).
                        // (the element-wise mask exists only in the masked instantiation,
                        // chosen once per tile)
                        if (masked)
                            exp_half_any<BF16, true, FP8V>(hi, 64 * hv, rel_lo, rel_hi, sc, neg_m, acc, p_addr, p8_addr);
                        else
                            exp_half_any<BF16, false, FP8V>(hi, 64, rel_lo, rel_hi, sc, neg_m, acc, p_addr, p8_addr);
                        if (one_half) {
                            // zeros for the other half's P (16-bit pairs: 32 columns;
                            // e5m2 quads: 16 columns)
                            if constexpr (FP8V) {
                                tmem_st16_zero(p8_addr + 16 * (1 - hv));
                            } else {
                                tmem_st16_zero(p_addr + 32 * (1 - hv));
                                tmem_st16_zero(p_addr + 32 * (1 - hv) + 16);
                            }
                        } else {
                            uint32_t lo[64];
                            tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(lo));
                            tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(lo + 32));
                            tmem_wait_ld();
                            if constexpr (C::SEP) {
                                // last read of this S: the MMA warp may overwrite it now
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0) mbar_arrive(bar(C::B_SFREE + wg));
                            }
                            if (masked)
                                exp_half_any<BF16, true, FP8V>(lo, 0, rel_lo, rel_hi, sc, neg_m, acc, p_addr, p8_addr);
                            else
                                exp_half_any<BF16, false, FP8V>(lo, 0, rel_lo, rel_hi, sc, neg_m, acc, p_addr, p8_addr);
                        }
                    }

                }
                acc[0] = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
                l = l * alpha + (acc[0].x + acc[0].y);

                if (__any_sync(0xffffffffu, rescale)) {
                    // O must hold every earlier P.V before it is rescaled.  In pair
                    // mode the S-ready commit already covered it; in single mode
                    // the previous tile's P.V used the other buffer.
                    if constexpr (!PAIR) ok = wait_pv(b ^ 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t o_addr = tmem + lane_off + C::o_col(PAIR ? wg : 0);
                    if constexpr (FP8V) {
                        // (the exact running max rescales on most tiles: 64 columns
                        // per TMEM round trip)
#pragma unroll 1
                        for (int c = 0; c < D / 32; c += 2) {
                            uint32_t r0[32], r1[32];
                            tmem_ld32(o_addr + 32 * c, r0);
                            tmem_ld32(o_addr + 32 * c + 32, r1);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                r0[e] = __float_as_uint(__uint_as_float(r0[e]) * alpha);
                                r1[e] = __float_as_uint(__uint_as_float(r1[e]) * alpha);
                            }
                            tmem_st32(o_addr + 32 * c, r0);
                            tmem_st32(o_addr + 32 * c + 32, r1);
                        }
                    } else {
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t raw[32];
                            tmem_ld32(o_addr + 32 * c, raw);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                raw[e] = __float_as_uint(__uint_as_float(raw[e]) * alpha);
                            tmem_st32(o_addr + 32 * c, raw);
                        }
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_PFULL + b));
                made.inc(b);
            }
            if (!ok) break;
            // ------------------------------------------------ epilogue: O / l, lse
            if (PAIR) {
                ok = wait_pv(wg);
            } else {
                ok = wait_pv(0) && wait_pv(1);
            }
            if (!ok) break;
            tc_fence_after();
            const float inv_l = 1.f / l;
            const uint32_t o_addr = tmem + lane_off + C::o_col(PAIR ? wg : 0);
            if (!dep) {
                griddep_wait();
                dep = true;
            }
            if constexpr (C::OSTAGE) {
                // Per 64 columns: the row's 16-byte chunks go to the warp's slab in
                // the 128-byte swizzled layout of the O map's 64 x 32 box (chunk
                // index XOR row mod 8: each store instruction covers all banks),
                // then one lane stores the warp's 32 rows; rows past L and columns
                // past d_out lie outside the map and are not written.
                const uint32_t slab = s_base + C::OFF_OST + static_cast<uint32_t>(warp) * C::OST_WARP_BYTES;
                const int row0 = qt * BM + wq * 32;
#pragma unroll 1
                for (int hc = 0; hc < D / 64; ++hc) {
                    if (lane == 0) bulk_wait_read0();     // the slab's previous store has read it
                    __syncwarp();
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        uint32_t raw[32];
                        tmem_ld32(o_addr + 64 * hc + 32 * c, raw);
                        tmem_wait_ld();
                        uint32_t w16[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w16[e] = pack2<BF16>(__uint_as_float(raw[2 * e]) * inv_l,
                                                 __uint_as_float(raw[2 * e + 1]) * inv_l);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            const uint32_t chunk = static_cast<uint32_t>(4 * c + v4);
                            st_shared_v4(slab + static_cast<uint32_t>(lane) * 128u + ((chunk ^ (lane & 7u)) << 4),
                                         w16[4 * v4], w16[4 * v4 + 1], w16[4 * v4 + 2], w16[4 * v4 + 3]);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && row0 < p.L && 64 * hc < p.d_out) {
                        tma_store_3d(&tmap_o, slab, 64 * hc, row0, U.bh);
                        bulk_commit();
                    }
                }
            } else {
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.o) +
                                                       ((static_cast<size_t>(U.bh) * p.L + i) * p.d_out) * 2);
#pragma unroll 1
                for (int c = 0; c < D / 32 && 32 * c < p.d_out; ++c) {
                    uint32_t raw[32];
                    tmem_ld32(o_addr + 32 * c, raw);
                    tmem_wait_ld();
                    uint32_t w16[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w16[e] = pack2<BF16>(__uint_as_float(raw[2 * e]) * inv_l,
                                             __uint_as_float(raw[2 * e + 1]) * inv_l);
                    if (row_valid) {
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            if (32 * c + 8 * v4 < p.d_out)
                                dst[c * 4 + v4] = make_uint4(w16[4 * v4], w16[4 * v4 + 1], w16[4 * v4 + 2],
                                                             w16[4 * v4 + 3]);
                    }
                }
            }
            if (row_valid && p.lse != nullptr) {
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                p.lse[static_cast<size_t>(U.bh) * p.L + i] =
                    (m_use + lg2_approx(l)) * 0.69314718055994530942f;
            }
            tc_fence_before();
        }
        // staged O: the last stores complete before the CTA's shared memory goes
        if constexpr (C::OSTAGE) {
            if (lane == 0) bulk_wait0();
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == C::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace attn
