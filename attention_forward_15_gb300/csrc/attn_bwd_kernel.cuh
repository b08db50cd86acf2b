// Fused attention backward for sm_103a (GB300): gradients dQ, dK, dV of the
// forward in attn_fwd_kernel.cuh for an output gradient dO, from the saved
// per-row log-sum-exp (the "Fused Attention" page keeps q, k, v, O and that
// statistic for a backward it does not define; this is the chain rule through
// the softmax):
//
//   P    = exp(sm_scale q_i.k_j - lse_i)           (zero outside the mask)
//   Di   = dO_i . O_i
//   dV_j = sum_i P_ij dO_i          dP_ij = dO_i . v_j
//   dS_ij = P_ij (dP_ij - Di)
//   dQ_i = sm_scale sum_j dS_ij k_j     dK_j = sm_scale sum_i dS_ij q_i
//
// Three kernels, no atomics (results are deterministic):
//   * attn_bwd_prep_kernel: Di per row, and per-head copies of -lse*log2(e)
//     and -Di padded to whole 128-row tiles (padding rows: -inf and 0, so that
//     rows past L give P = 0 wherever they are read);
//   * attn_bwd_kernel<D, BF16, false> ("dK/dV"): one CTA per (head, key tile);
//     K and V of the tile stay in shared memory while the query tiles that
//     attend it stream through a ring; per query tile
//         S^T = K Q^T, dP^T = V dO^T       (tcgen05, fp32 in tensor memory)
//         P^T, dS^T in the compute warps   (one thread per key row and 32 columns)
//         dV += P^T dO, dK += dS^T Q       (A operand from tensor memory)
//   * attn_bwd_kernel<D, BF16, true> ("dQ"): one CTA per (head, query tile);
//     Q and dO stay while the attended key tiles stream; per key tile
//         S = Q K^T, dP = dO V^T, dS in the compute warps (one thread per query
//         row), dQ += dS K.
// Both are one template: a CTA holds a "fixed" pair of tiles (F0, F1) and
// streams pairs (R0, R1); the products are S = F0 R0^T and dP = F1 R1^T in
// either kernel, then (dK/dV) ACC0 += P R1 and, in both, ACC1 += dS R0.
//
// Each streamed tile is taken as two halves of 64 rows, each with S and dP
// buffers of its own in tensor memory, so the MMA pipe computes one half's
// products while the compute warps work on the other:
//   S_0 | dP_0 | S_1 | dP_1 (64 columns each) | ACC0 (D) | ACC1 (D).
// All four compute warpgroups take each half in turn, 16 columns a group; a
// group writes its P (16-bit pairs) over the first 8 of its S columns and its
// dS over the first 8 of its dP columns, once read; a half's next S and dP
// are issued after the products that read its P and dS, on the same in-order
// MMA pipe.  D is 64 or 128 (256 + 2D columns), or 256: then the fixed pair
// fills 128 KB of shared memory, the ring holds one 64-row half of the streamed
// pair at a time, and dK/dV runs two CTAs per key tile, each accumulating one
// half of the head dim (256 + 2 x 128 columns; dQ: 256 + 256).
#pragma once

#include "attn_fwd_kernel.cuh"

namespace attn {

struct BwdParams {
    const void *o;           // prep: forward output [BH, L, d_out] 16-bit
    const void *dout;        // prep: output gradient [BH, L, d_out] 16-bit
    const float *lse;        // prep: forward lse [BH, L] (natural log)
    float *nlse2;            // [BH, n_pad]: -lse * log2(e), -inf past L
    float *ndelta;           // [BH, n_pad]: -Di, 0 past L
    void *g0;                // dK/dV: dK, dQ: dQ   [BH, L, d_out] 16-bit
    void *g1;                // dK/dV: dV           [BH, L, d_out] 16-bit
    unsigned int *status;
    int BH, L, mask, bs;
    int n_t;                 // 128-row tiles per head
    int n_pad;               // n_t * 128
    float scale;             // sm_scale
    float scale_log2;        // sm_scale * log2(e)
    int d_out;               // head dim in memory (<= D of the kernel)
    int inject;              // test hook: 1 = the producer issues no copies, so every
                             // consumer's bounded wait runs out (0 in normal use)
};

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

// ------------------------------------------------------------------ prep

// Di = sum_d dO[i,d] O[i,d] (fp32) for every row of every head, stored as -Di
// with -lse * log2(e) beside it (negated so that the tile kernels take them
// with one packed fma and one packed add), padded to n_pad rows.  Eight
// threads per row, 16 bytes each per step, reduced by shuffles; grid-stride
// over rows.
template <bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdParams p) {
    griddep_wait();
    griddep_launch_dependents();
    const int sub = threadIdx.x & 7;
    const long long rows = static_cast<long long>(p.BH) * p.n_pad;
    const long long stride = static_cast<long long>(gridDim.x) * (blockDim.x / 8);
    for (long long r = static_cast<long long>(blockIdx.x) * (blockDim.x / 8) + (threadIdx.x >> 3); r < rows;
         r += stride) {
        const int bh = static_cast<int>(r / p.n_pad);
        const int i = static_cast<int>(r % p.n_pad);
        float acc = 0.f;
        if (i < p.L) {
            const size_t base = (static_cast<size_t>(bh) * p.L + i) * p.d_out;
            const uint4 *o4 = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.o) + base);
            const uint4 *g4 = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.dout) + base);
            for (int c = sub; c < p.d_out / 8; c += 8) {
                const uint4 a = o4[c], b = g4[c];
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x = unpack2<BF16>(aw[e]), y = unpack2<BF16>(bw[e]);
                    acc = fmaf(x.x, y.x, acc);
                    acc = fmaf(x.y, y.y, acc);
                }
            }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        if (sub == 0) {
            p.ndelta[r] = i < p.L ? -acc : 0.f;
            p.nlse2[r] = i < p.L ? p.lse[static_cast<size_t>(bh) * p.L + i] * -1.4426950408889634f : -INFINITY;
        }
    }
}

// ------------------------------------------------------------------ dK/dV and dQ

template <int D, bool DQ>
struct BwdCfg {
    static constexpr int CHUNKS = D / 64;               // 128-byte-wide TMA boxes per row
    static constexpr int CHUNK_BYTES = 128 * 128;       // one box of a fixed tile: 128 rows
    static constexpr int TILE_BYTES = 128 * D * 2;
    // D = 256: the fixed pair alone takes 128 KB of shared memory, so the ring
    // holds the 64-row halves of the streamed tiles (one stage of the two
    // operands, 64 KB) instead of whole tiles.
    static constexpr bool HALF_RING = D == 256;
    static constexpr int RCHUNK_BYTES = HALF_RING ? 64 * 128 : CHUNK_BYTES;  // one box of a ring operand
    static constexpr int RTILE_BYTES = HALF_RING ? TILE_BYTES / 2 : TILE_BYTES;
    static constexpr int NS = HALF_RING ? 1 : (D == 64 ? 3 : 2);   // ring stages of streamed pairs
    // dK/dV at D = 256: the two accumulators would need 2 x 256 columns of tensor
    // memory next to S and dP, so each CTA keeps half of the head dim of dK and
    // dV (two CTAs per key tile, both computing S and dP over the whole head dim)
    static constexpr bool DSPLIT = HALF_RING && !DQ;
    static constexpr int DA = DSPLIT ? D / 2 : D;        // accumulator width (columns)
    // four compute warpgroups (group w takes 16 of the 64 rows of each half of
    // every streamed tile), a TMA warp and an MMA warp
    static constexpr int THREADS = 576;
    static constexpr int WARP_TMA = 16, WARP_MMA = 17;
    static constexpr int VEC_ROWS = HALF_RING ? 64 : 128;    // rows of a ring entry
    static constexpr int VEC_BYTES = DQ ? 0 : 2 * VEC_ROWS * 4;   // -lse2 and -Di of those rows
    static constexpr int OFF_FIX = 0;                        // F0 | F1
    static constexpr int OFF_RING = 2 * TILE_BYTES;          // NS x (R0 | R1)
    static constexpr int OFF_VEC = OFF_RING + NS * 2 * RTILE_BYTES;
    static constexpr int OFF_BAR = OFF_VEC + NS * VEC_BYTES;
    static constexpr int B_FIX = 0, B_FULL = 1, B_EMPTY = 1 + NS, B_SFULL = 1 + 2 * NS;   // SFULL, PFULL: one per half
    static constexpr int B_PFULL = B_SFULL + 2, B_DONE = B_PFULL + 2, B_DRAIN = B_DONE + 1;
    static constexpr int B_FIXT = B_DRAIN + 1;             // FIX_TMEM: fixed pair copied to TMEM
    static constexpr int NBAR = B_FIXT + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;     // [0]: TMEM base, [1]: abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr int HALF_BYTES = 64 * 128;          // 64 rows of a 128-byte-wide box
    __device__ static constexpr uint32_t col_s(int h) { return 128u * static_cast<uint32_t>(h); }
    __device__ static constexpr uint32_t col_dp(int h) { return 128u * static_cast<uint32_t>(h) + 64u; }
    // ACC0 (dV, dK/dV only) and ACC1 (dK or dQ) after the S and dP buffers
    static constexpr uint32_t COL_ACC0 = 256, COL_ACC1 = DQ ? 256 : 256 + DA;
    // FIX_TMEM (D = 64, where the columns allow it): the fixed pair also sits in
    // TMEM (16-bit pairs, row = lane), so S and dP take their A operand from
    // there and read only the streamed half-tile from shared memory (a
    // shared/shared N = 64 product is bound by shared-memory bandwidth).
    static constexpr bool FIX_TMEM = D == 64;
    static constexpr uint32_t COL_F0 = COL_ACC1 + DA, COL_F1 = COL_F0 + D / 2;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(D == 64 || D == 128 || D == 256, "backward head dim");
    static_assert(COL_ACC1 + DA <= TMEM_COLS, "tensor memory budget");
    static_assert(!FIX_TMEM || COL_F1 + D / 2 <= TMEM_COLS, "tensor memory budget (fixed pair)");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Streamed-tile range [lo, hi) of a CTA whose fixed tile is f: for dK/dV the
// query tiles that attend key tile f, for dQ the key tiles query tile f
// attends (tiles wholly outside the mask are left out).
__device__ __forceinline__ void bwd_range(const BwdParams &p, bool dq, int f, int &lo, int &hi) {
    if (p.mask == kMaskDense) {
        lo = 0;
        hi = p.n_t;
    } else if (p.mask == kMaskCausal) {
        lo = dq ? 0 : f;
        hi = dq ? f + 1 : p.n_t;
    } else {
        // blocks are symmetric: the tiles meeting the blocks of tile f
        const int r0 = f * 128;
        const int r1 = min(r0 + 128, p.L);
        const int blo = (r0 / p.bs) * p.bs;
        const int bhi = ((r1 - 1) / p.bs + 1) * p.bs;
        lo = blo / 128;
        hi = (bhi + 127) / 128;
    }
}

// dS (and P) of one chunk of NE columns: rows are this thread's TMEM lane,
// columns c0..c0+NE-1 of the tile.  S, dP: fp32 raw scores and dP of the chunk.  The
// negated lse2 and Di come per row (dQ: nl_row, nd_row) or per column (dK/dV:
// the shared-memory vectors from entry vc0 on, read four at a time); packed
// fp32x2 arithmetic as in the forward; `keep` masks (row, column).
template <bool BF16, bool DQ, bool MASKED, int NE>
__device__ __forceinline__ void bwd_chunk(const uint32_t (&S)[NE], const uint32_t (&dP)[NE], float sc,
                                          float nl_row, float nd_row, const float *col_nl,
                                          const float *col_nd, int c0, int vc0, int mask, int bs, int L,
                                          int row_idx, int col_base, uint32_t (&pk)[NE / 2],
                                          uint32_t (&dk)[NE / 2]) {
    static_assert(NE % 4 == 0, "bwd_chunk: whole float4s of the column vectors");
    const float2 sc2 = make_float2(sc, sc);
#pragma unroll
    for (int e = 0; e < NE / 2; ++e) {
        float2 nl, nd;
        if constexpr (DQ) {
            nl = make_float2(nl_row, nl_row);
            nd = make_float2(nd_row, nd_row);
        } else {
            const float4 a = reinterpret_cast<const float4 *>(col_nl + vc0)[e >> 1];
            const float4 b = reinterpret_cast<const float4 *>(col_nd + vc0)[e >> 1];
            nl = (e & 1) ? make_float2(a.z, a.w) : make_float2(a.x, a.y);
            nd = (e & 1) ? make_float2(b.z, b.w) : make_float2(b.x, b.y);
        }
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(S[2 * e]), __uint_as_float(S[2 * e + 1])), sc2, nl);
        float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        if constexpr (MASKED) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // (query, key) of this element; keys past L are zero rows whose
                // p could overflow when lse is very negative, so they are cut too
                const int c = c0 + 2 * e + h;
                const int qi = DQ ? row_idx : col_base + c;
                const int kj = DQ ? col_base + c : row_idx;
                bool keep = kj < L;
                if (mask == kMaskCausal) keep = keep && kj <= qi;
                else if (mask == kMaskBlock) keep = keep && (kj / bs) == (qi / bs);
                if (!keep) {
                    if (h == 0) pp.x = 0.f;
                    else pp.y = 0.f;
                }
            }
        }
        const float2 ds = __fmul2_rn(
            pp, __fadd2_rn(make_float2(__uint_as_float(dP[2 * e]), __uint_as_float(dP[2 * e + 1])), nd));
        pk[e] = pack2<BF16>(pp.x, pp.y);
        dk[e] = pack2<BF16>(ds.x, ds.y);
    }
}

template <int D, bool BF16, bool DQ>
__global__ void __launch_bounds__(BwdCfg<D, DQ>::THREADS, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_f0, const __grid_constant__ CUtensorMap tm_f1,
                const __grid_constant__ CUtensorMap tm_r0, const __grid_constant__ CUtensorMap tm_r1,
                const __grid_constant__ CUtensorMap tm_g0, const __grid_constant__ CUtensorMap tm_g1,
                const BwdParams p) {
    using C = BwdCfg<D, DQ>;
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

    // unit of this CTA: (head, fixed tile).  Causal: heaviest fixed tiles first
    // across all heads; otherwise head-major, so that CTAs running together
    // stream the same head's tiles (shared in L2)
    // (DSPLIT: the two CTAs of a key tile are neighbours; dc = head-dim half)
    const unsigned bid = C::DSPLIT ? blockIdx.x >> 1 : blockIdx.x;
    const int dc = C::DSPLIT ? static_cast<int>(blockIdx.x & 1u) : 0;
    const bool head_major = p.mask != kMaskCausal;
    const int bh = head_major ? static_cast<int>(bid / static_cast<unsigned>(p.n_t))
                              : static_cast<int>(bid % static_cast<unsigned>(p.BH));
    const int rank = head_major ? static_cast<int>(bid % static_cast<unsigned>(p.n_t))
                                : static_cast<int>(bid / static_cast<unsigned>(p.BH));
    const int f = (p.mask == kMaskCausal && DQ) ? p.n_t - 1 - rank : rank;
    int lo, hi;
    bwd_range(p, DQ, f, lo, hi);
    const int n = hi - lo;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_FIX), 1);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar(C::B_FULL + s), 1);
            mbar_init(bar(C::B_EMPTY + s), 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(bar(C::B_SFULL + h), 1);
            mbar_init(bar(C::B_PFULL + h), 16);   // one arrival per compute warp
        }
        mbar_init(bar(C::B_DONE), 1);
        mbar_init(bar(C::B_DRAIN), 1);
        mbar_init(bar(C::B_FIXT), 8);   // FIX_TMEM: one arrival per copying warp
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == C::WARP_TMA && lane == 0) {
        tma_prefetch_desc(&tm_f0);
        tma_prefetch_desc(&tm_f1);
        tma_prefetch_desc(&tm_r0);
        tma_prefetch_desc(&tm_r1);
    }
    if (warp == C::WARP_MMA) {
        tmem_alloc(s_base + C::OFF_MISC, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();
    griddep_launch_dependents();
    constexpr uint32_t tmem = 0;
    const bool tmem_ok = misc[0] == 0u;
    if (!tmem_ok && threadIdx.x == 0) atomicCAS(p.status, 0u, kStatusTmem);
    const int nn = tmem_ok ? n : 0;

    auto wait_warp = [&](uint32_t bar_addr, uint32_t parity, unsigned site) -> bool {
        const bool r = wait_bar(bar_addr, parity, ctl, site);
        return __all_sync(0xffffffffu, r);
    };

    if (warp == C::WARP_TMA) {
        // ================================================================ TMA producer
        uint32_t issued = 0;          // streamed stages issued
        bool fix_issued = false;
        bool ok = p.inject != 1;
        if (ok && nn > 0) {
            mbar_arrive_expect_tx(bar(C::B_FIX), 2 * C::TILE_BYTES);
            for (int c = 0; c < C::CHUNKS; ++c) {
                tma_load_3d(s_base + C::OFF_FIX + c * C::CHUNK_BYTES, &tm_f0, c * 64, f * 128, bh, bar(C::B_FIX));
                tma_load_3d(s_base + C::OFF_FIX + C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_f1, c * 64, f * 128, bh,
                            bar(C::B_FIX));
            }
            fix_issued = true;
        }
        // ring entries: whole streamed tiles, or (HALF_RING) their 64-row halves in turn
        constexpr int PER_TILE = C::HALF_RING ? 2 : 1;
        for (int q = 0; q < PER_TILE * nn && ok; ++q) {
            const int s = q % C::NS;
            ok = wait_warp(bar(C::B_EMPTY + s), ((q / C::NS) & 1) ^ 1, kSiteKvEmpty);
            if (!ok) break;
            const int j = lo + q / PER_TILE;
            const int row0 = j * 128 + (q % PER_TILE) * 64;
            mbar_arrive_expect_tx(bar(C::B_FULL + s), 2 * C::RTILE_BYTES + C::VEC_BYTES);
            const uint32_t dst = s_base + C::OFF_RING + s * 2 * C::RTILE_BYTES;
            for (int c = 0; c < C::CHUNKS; ++c) {
                tma_load_3d(dst + c * C::RCHUNK_BYTES, &tm_r0, c * 64, row0, bh, bar(C::B_FULL + s));
                tma_load_3d(dst + C::RTILE_BYTES + c * C::RCHUNK_BYTES, &tm_r1, c * 64, row0, bh,
                            bar(C::B_FULL + s));
            }
            if constexpr (!DQ) {
                const size_t off = static_cast<size_t>(bh) * p.n_pad + static_cast<size_t>(row0);
                const uint32_t vdst = s_base + C::OFF_VEC + s * C::VEC_BYTES;
                bulk_load_1d(vdst, p.nlse2 + off, C::VEC_ROWS * 4, bar(C::B_FULL + s));
                bulk_load_1d(vdst + C::VEC_ROWS * 4, p.ndelta + off, C::VEC_ROWS * 4, bar(C::B_FULL + s));
            }
            ++issued;
        }
        if (*ctl.abort_flag) {
            // stopping early: the copies already issued land before shared memory goes away
            if (fix_issued) wait_slow(bar(C::B_FIX), 0, ctl, kSiteDrain, false);
            const uint32_t first = issued > static_cast<uint32_t>(C::NS) ? issued - C::NS : 0u;
            for (uint32_t t = first; t < issued; ++t)
                wait_slow(bar(C::B_FULL + t % C::NS), (t / C::NS) & 1u, ctl, kSiteDrain, false);
        }
        __syncwarp();
    } else if (warp == C::WARP_MMA) {
        // ================================================================ MMA issuer
        constexpr uint32_t IDESC_SS = idesc_f16_f32acc(BF16, 128, 64, false);
        constexpr uint32_t IDESC_ACC = idesc_f16_f32acc(BF16, 128, C::DA, true);
        const uint32_t f0 = s_base + C::OFF_FIX, f1 = f0 + C::TILE_BYTES;
        // X = A B^T over the head dim for 64 rows of B: both K-major, k-step kk
        // = head-dim columns [16kk, 16kk+16): box kk/4 (fixed A: CHUNK_BYTES apart,
        // ring B: RCHUNK_BYTES apart), 32-byte offset kk%4.
        // (FIX_TMEM: A is the fixed tile's copy in TMEM at column a_tcol)
        auto issue_fs = [&](uint32_t a_tcol, uint32_t b, uint32_t dcol) {
            const uint32_t a = tmem + a_tcol;
            mma_ts_x4(tmem + dcol, a, a + 8, a + 16, a + 24, sdesc_sw128(b, 16, 1024), 2, IDESC_SS, 0u);
        };
        auto issue_ss = [&](uint32_t a, uint32_t b, uint32_t dcol) {
#pragma unroll
            for (int c = 0; c < C::CHUNKS; ++c)   // four k-steps (32 bytes apart) per 64-column box
                mma_ss_x4(tmem + dcol, sdesc_sw128(a + c * C::CHUNK_BYTES, 16, 1024),
                          sdesc_sw128(b + c * C::RCHUNK_BYTES, 16, 1024), 2, 2, IDESC_SS, c > 0 ? 1u : 0u);
        };
        // ACC += A(TMEM, 16-bit pairs) B over 64 rows of B, B MN-major: k-step kk
        // = rows [16kk, 16kk+16); its 64-column boxes are RCHUNK_BYTES apart (DSPLIT:
        // starting at the head-dim half dc).  The A pairs of rows [16kk, 16kk+16)
        // sit at columns 16kk..16kk+7 of the half.
        auto issue_acc = [&](uint32_t acol, uint32_t b, uint32_t dcol, bool accumulate) {
            const uint64_t bd =
                sdesc_sw128(b + static_cast<uint32_t>(dc * (C::DA / 64) * C::RCHUNK_BYTES), C::RCHUNK_BYTES, 1024);
            const uint32_t a = tmem + acol;
            mma_ts_x4(tmem + dcol, a, a + 16, a + 32, a + 48, bd, 128, IDESC_ACC, accumulate ? 1u : 0u);
        };
        // S_h and dP_h of the tile in ring stage `stage`
        auto issue_half = [&](int stage, int h) {
            const uint32_t r0 = s_base + C::OFF_RING + stage * 2 * C::TILE_BYTES + h * C::HALF_BYTES;
            if constexpr (C::FIX_TMEM) {
                issue_fs(C::COL_F0, r0, C::col_s(h));
                issue_fs(C::COL_F1, r0 + C::TILE_BYTES, C::col_dp(h));
            } else {
                issue_ss(f0, r0, C::col_s(h));
                issue_ss(f1, r0 + C::TILE_BYTES, C::col_dp(h));
            }
            mma_commit(bar(C::B_SFULL + h));
        };
        bool ok = nn > 0;
        if (ok) ok = wait_warp(bar(C::B_FIX), 0, kSiteQFull);
        if constexpr (C::FIX_TMEM) {
            if (ok) ok = wait_warp(bar(C::B_FIXT), 0, kSiteQFull);
        }
        if constexpr (C::HALF_RING) {
            // One ring entry per 64-row half: its S and dP, then (once the half's
            // compute warps have written P and dS) its two accumulations, which
            // free the entry for the next half.
            for (int q = 0; q < 2 * nn && ok; ++q) {
                const int t = q >> 1, h = q & 1, s = q % C::NS;
                ok = wait_warp(bar(C::B_FULL + s), (q / C::NS) & 1, kSiteKvFullK);
                if (!ok) break;
                tc_fence_after();
                const uint32_t r0 = s_base + C::OFF_RING + s * 2 * C::RTILE_BYTES;
                const uint32_t r1 = r0 + C::RTILE_BYTES;
                issue_ss(f0, r0, C::col_s(h));
                issue_ss(f1, r1, C::col_dp(h));
                mma_commit(bar(C::B_SFULL + h));
                ok = wait_warp(bar(C::B_PFULL + h), t & 1, kSitePFull);
                if (!ok) break;
                tc_fence_after();
                if constexpr (!DQ) issue_acc(C::col_s(h), r1, C::COL_ACC0, q > 0);   // dV += P^T dO
                issue_acc(C::col_dp(h), r0, C::COL_ACC1, q > 0);                       // dK += dS^T Q | dQ += dS K
                mma_commit(bar(C::B_EMPTY + s));
            }
            ok = ok && nn > 0;
        } else {
        if (ok) ok = wait_warp(bar(C::B_FULL + 0), 0, kSiteKvFullK);
        if (ok) {
            tc_fence_after();
            issue_half(0, 0);
            issue_half(0, 1);
        }
        for (int t = 0; t < nn && ok; ++t) {
            const int s = t % C::NS;
            const int s2 = (t + 1) % C::NS;
#pragma unroll 1
            for (int h = 0; h < 2 && ok; ++h) {
                ok = wait_warp(bar(C::B_PFULL + h), t & 1, kSitePFull);
                if (!ok) break;
                tc_fence_after();
                const uint32_t r0 = s_base + C::OFF_RING + s * 2 * C::TILE_BYTES + h * C::HALF_BYTES;
                const uint32_t r1 = r0 + C::TILE_BYTES;
                const bool acc = t > 0 || h > 0;
                if constexpr (!DQ) issue_acc(C::col_s(h), r1, C::COL_ACC0, acc);   // dV += P^T dO
                issue_acc(C::col_dp(h), r0, C::COL_ACC1, acc);                       // dK += dS^T Q | dQ += dS K
                if (h == 1) mma_commit(bar(C::B_EMPTY + s));
                if (t + 1 < nn) {
                    if (h == 0) {
                        ok = wait_warp(bar(C::B_FULL + s2), ((t + 1) / C::NS) & 1, kSiteKvFullK);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    issue_half(s2, h);
                }
            }
        }
        }   // whole-tile ring
        if (ok && nn > 0) mma_commit(bar(C::B_DONE));
        // every MMA (and the arrivals its commits make) done before the CTA
        // frees tensor memory and exits
        mma_commit(bar(C::B_DRAIN));
        wait_slow(bar(C::B_DRAIN), 0, ctl, kSiteDrain, false);
        __syncwarp();
    } else {
        // ================================================================ compute warps
        // group wg takes columns [16wg, 16wg+16) of each half of every streamed
        // tile, half 0 then half 1; each thread owns one TMEM lane, i.e. one row
        // of the fixed tile
        const int wg = warp >> 2;
        const int row = (warp & 3) * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const int row_idx = f * 128 + row;                 // query (dQ) or key (dK/dV) index
        const float sc = p.scale_log2;
        float row_nl = 0.f, row_nd = 0.f;
        if constexpr (DQ) {
            row_nl = p.nlse2[static_cast<size_t>(bh) * p.n_pad + row_idx];
            row_nd = p.ndelta[static_cast<size_t>(bh) * p.n_pad + row_idx];
        }
        bool ok = true;
        if constexpr (C::FIX_TMEM) {
            // warps 0-3 copy F0, warps 4-7 F1: each thread its row, the eight
            // 16-byte chunks (128-byte swizzle: chunk index XOR row mod 8) as 32
            // words of 16-bit pairs, k-step kk at columns 8kk..8kk+7
            if (warp < 8 && nn > 0) {
                ok = wait_warp(bar(C::B_FIX), 0, kSiteQFull);
                if (ok) {
                    const int which = warp >> 2;
                    const uint32_t src = s_base + C::OFF_FIX + which * C::TILE_BYTES + static_cast<uint32_t>(row) * 128u;
                    uint32_t w[32];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 v = ld_shared_v4(src + ((static_cast<uint32_t>(c) ^ (static_cast<uint32_t>(row) & 7u)) << 4));
                        w[4 * c] = v.x;
                        w[4 * c + 1] = v.y;
                        w[4 * c + 2] = v.z;
                        w[4 * c + 3] = v.w;
                    }
                    tmem_st32(tmem + lane_off + (which ? C::COL_F1 : C::COL_F0), w);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::B_FIXT));
                }
            }
        }
        for (int t = 0; t < nn && ok; ++t) {
            const int j = lo + t;
            // tiles that cross the mask, and (dQ) a ragged last key tile
            const bool masked = (p.mask == kMaskCausal && j == f) || (p.mask == kMaskBlock && (p.bs % 128) != 0) ||
                                (DQ && (j + 1) * 128 > p.L);
#pragma unroll 1
            for (int h = 0; h < 2 && ok; ++h) {
                // ring entry of this half: the tile's (whole-tile ring) or the
                // half's own (HALF_RING, whose vectors then start at the half's rows)
                const int s = C::HALF_RING ? (2 * t + h) % C::NS : t % C::NS;
                const float *vec = reinterpret_cast<const float *>(smem + C::OFF_VEC + s * C::VEC_BYTES);
                const uint32_t cs = tmem + lane_off + C::col_s(h) + 16 * wg;    // this group's S columns
                const uint32_t cd = tmem + lane_off + C::col_dp(h) + 16 * wg;   // and dP columns
                ok = wait_warp(bar(C::B_SFULL + h), t & 1, kSiteSFull);
                if (!ok) break;
                tc_fence_after();
                uint32_t sv[16], dpv[16];
                tmem_ld16(cs, sv);
                tmem_ld16(cd, dpv);
                tmem_wait_ld();
                uint32_t pk[8], dk[8];
                const int c0 = 64 * h + 16 * wg;              // column of the chunk in the tile
                const int vc0 = C::HALF_RING ? 16 * wg : c0;
                if (masked)
                    bwd_chunk<BF16, DQ, true, 16>(sv, dpv, sc, row_nl, row_nd, vec, vec + C::VEC_ROWS, c0, vc0,
                                                  p.mask, p.bs, p.L, row_idx, j * 128, pk, dk);
                else
                    bwd_chunk<BF16, DQ, false, 16>(sv, dpv, sc, row_nl, row_nd, vec, vec + C::VEC_ROWS, c0, vc0,
                                                   p.mask, p.bs, p.L, row_idx, j * 128, pk, dk);
                // P and dS to the first 8 of this group's S and dP columns, which
                // it has read by now
                if constexpr (!DQ) tmem_st8(cs, pk);
                tmem_st8(cd, dk);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_PFULL + h));
            }
        }
        if (ok && nn > 0) ok = wait_warp(bar(C::B_DONE), 0, kSiteODone);
        if (ok && nn > 0) {
            tc_fence_after();
            // 32-column jobs: ACC1 (dK or dQ, times sm_scale) to g0, and (dK/dV)
            // ACC0 (dV) to g1, dealt round-robin to the four groups; the
            // accumulators hold head-dim columns [dc * DA, dc * DA + DA).  A job's
            // 32 rows of the warp go through a 2 KB slab of the fixed-tile area
            // (free once the last MMA is done) in the 64-byte swizzled layout of
            // the output map's 32 x 32 box (16-byte chunk index XOR (row / 2) mod
            // 4), then one lane stores them; rows past L and columns past d_out
            // lie outside the map and are not written.
            constexpr int NJ = (DQ ? 1 : 2) * (C::DA / 32);
            static_assert(16 * 2048 <= 2 * C::TILE_BYTES, "output slabs fit the fixed-tile area");
            const uint32_t slab = s_base + C::OFF_FIX + static_cast<uint32_t>(warp) * 2048u;
            const int row0 = f * 128 + (warp & 3) * 32;
#pragma unroll 1
            for (int jb = wg; jb < NJ; jb += 4) {
                const bool to_g0 = jb < C::DA / 32;
                const int c = jb % (C::DA / 32);
                const int col0 = dc * C::DA + 32 * c;           // first head-dim column of the job
                if (col0 >= p.d_out) continue;
                const uint32_t acol = to_g0 ? C::COL_ACC1 : C::COL_ACC0;
                const float mul = to_g0 ? p.scale : 1.f;
                uint32_t raw[32];
                tmem_ld32(tmem + lane_off + acol + 32 * c, raw);
                tmem_wait_ld();
                uint32_t w16[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w16[e] = pack2<BF16>(__uint_as_float(raw[2 * e]) * mul, __uint_as_float(raw[2 * e + 1]) * mul);
                if (lane == 0) bulk_wait_read0();     // the slab's previous store has read it
                __syncwarp();
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    st_shared_v4(slab + static_cast<uint32_t>(lane) * 64u +
                                     ((static_cast<uint32_t>(v4) ^ ((static_cast<uint32_t>(lane) >> 1) & 3u)) << 4),
                                 w16[4 * v4], w16[4 * v4 + 1], w16[4 * v4 + 2], w16[4 * v4 + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && row0 < p.L) {
                    tma_store_3d(to_g0 ? &tm_g0 : &tm_g1, slab, col0, row0, bh);
                    bulk_commit();
                }
            }
        }
        // the output stores complete before the CTA's shared memory goes
        if (lane == 0) bulk_wait0();
        __syncwarp();
        tc_fence_before();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == C::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace attn
