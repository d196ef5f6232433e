// chain_dense_tc.cu -- chained composition for the gated delta rule on tcgen05.
//
// For one (request, layer, head) the combine step folds pool entries in order,
//     S <- exp(lambda_p) M_p S + S_p,
// one 128 x 128 x 128 product per step.  The product runs on the tensor cores
// in bf16 with both operands split three ways (x = hi + mid + lo, residual
// ~2^-27) and the six partial products down to order 2^-16 kept (~2^-24
// relative per product), which keeps the fp32 composition well inside 1e-5.
// The exact fp32 running state stays in the math warps' registers (row i of S
// on TMEM lane i, four warps per lane quarter, 32 columns each).
//
// Persistent: one CTA per SM walks its units (a unit is one chain; without a
// chain list it is one composition S = exp(lambda) M S_prev + S_C) step after
// step.  Warp 0 brings each M_p (lane 0) and S_p (lane 1) into shared memory by
// TMA (128-byte swizzle, so the row-per-lane reads are conflict-free); the math
// warps split M_p into one of two TMEM operand buffers -- the NEXT step's M_p
// while the current step's products run -- and split S into shared memory as
// the MN-major B operand.  The columns of S evolve independently, so the two
// 64-column halves run as two pipelines (their own math warps, barriers and MMA
// issuer, warps 1 and 18), sharing only the M_p operand.  Each unit's S_init comes
// through the M_p stage too (one more TMA fill, after the unit's first M_p, in
// flight during the previous unit's last products and update); the last update
// is written over S_p in its stage and leaves by TMA store.
// All global traffic of the state thus moves by TMA, none through per-thread
// row loads and stores.
#include "internal.cuh"
#include "sm100.cuh"

namespace hypic {
namespace {

using namespace sm100;

constexpr int kD = 128;
constexpr int kThreads = 608;           // warp 0: TMA, warps 1 and 18: MMA (one column half each), 2..17: math
constexpr int kMath = 512;
constexpr uint32_t kTa = 0;             // TMEM: A buffers at 0 and 192 (hi / mid / lo at +0, +64, +128)
constexpr uint32_t kTd = 384;           // D (128 columns)
constexpr int kBpart = 32768;           // one bf16 B tile: 128 k-rows x 128 n, 2 atoms of 64 n
constexpr int kMstage = 3 * kBpart;     // M_p stage, fp32, 4 boxes of 32 columns x 128 rows
constexpr int kSstage = kMstage + 65536; // S_p stage, same layout
constexpr int kCtl = kSstage + 65536;
constexpr int kSmem = kCtl + 256 + 1024;
static_assert(kSmem <= 232448, "fits in one SM's shared memory");

struct ChainCtrl {
    uint64_t mfull, mfree, sfull, sfree;
    uint64_t ops_ready[2], d_done[2];   // per column half: B half in shared memory / its products done
    uint64_t aready[2], afree[2];       // per A operand buffer: split into TMEM / read by both halves
    float rmax[2][16];                  // operator mode: the math warps' maxima, by renormalisation parity
    uint32_t tmem;
    int abort;
};

static_assert(sizeof(ChainCtrl) <= 256, "the control block fits its reserved bytes");

// Two fp32 values -> three packed bf16 pairs with x = hi + mid + lo (to ~2^-27 relative).
// (the residuals are exact, so the packed subtractions change no bit)
__device__ __forceinline__ void split3_pair(float x0, float x1, uint32_t &hi, uint32_t &mid, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    const uint64_t r = sub2(pk2(x0, x1), bf16x2_to_f32x2(hi));
    float r0, r1;
    upk2(r, r0, r1);
    const __nv_bfloat162 m = __floats2bfloat162_rn(r0, r1);
    mid = *reinterpret_cast<const uint32_t *>(&m);
    float q0, q1;
    upk2(sub2(r, bf16x2_to_f32x2(mid)), q0, q1);
    const __nv_bfloat162 l = __floats2bfloat162_rn(q0, q1);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Two fp32 values -> two packed bf16 pairs with x = hi + lo (to ~2^-17 relative).
__device__ __forceinline__ void split2_pair(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    float r0, r1;
    upk2(sub2(pk2(x0, x1), bf16x2_to_f32x2(hi)), r0, r1);
    const __nv_bfloat162 l = __floats2bfloat162_rn(r0, r1);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Steps of unit u (a chain of request r; one step without a chain list), clamped.
__device__ __forceinline__ int unit_steps(const ChainArgs &a, int64_t u, bool flag) {
    if (!a.chain_len) return 1;
    const int r = (int)(u / ((int64_t)a.n_layers * a.H));
    int n = a.chain_len[r];
    if (n < 0 || n > a.max_chain) {
        if (flag) flag_index_error(a.d_err);
        n = n < 0 ? 0 : a.max_chain;
    }
    return n;
}

// Pool row (entry, layer, head) of step c of unit u, clamped.
__device__ __forceinline__ int64_t step_entry(const ChainArgs &a, int64_t u, int c, bool flag) {
    const int64_t lhn = (int64_t)a.n_layers * a.H;
    const int r = (int)(u / lhn);
    const int64_t lh = u % lhn;
    int p = a.seg_idx ? a.seg_idx[(int64_t)r * a.max_chain + c] : (a.seg_first ? a.seg_first[r] + c : r);
    if (p < 0 || p >= a.P) {
        if (flag) flag_index_error(a.d_err);
        p = p < 0 ? 0 : a.P - 1;
    }
    return (int64_t)p * lhn + lh;
}

// OP: operator mode (ChainArgs::op), a compile-time switch so that the state's
// chain carries none of it.  NS: bf16 parts per operand, 3 (hi / mid / lo, six
// products: the fp32 compose) or 2 (hi / lo, three products, ~2^-17 per product:
// ChainArgs::two_way, for chains inside a scan whose inputs are bf16)
template <bool OP, int NS>
__global__ void __launch_bounds__(kThreads, 1)   // 19 warps: <= 96 registers per thread
    chain_dense_tc_kernel(const __grid_constant__ CUtensorMap tm_m, const __grid_constant__ CUtensorMap tm_s,
                          const __grid_constant__ CUtensorMap tm_i, const __grid_constant__ CUtensorMap tm_o,
                          const ChainArgs a, int64_t units) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align1024(smem_raw);
    ChainCtrl *ctl = reinterpret_cast<ChainCtrl *>(smem + kCtl);
    volatile int *abortp = &ctl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&ctl->mfull, 1);
        mbar_init(&ctl->mfree, kMath / 32);
        mbar_init(&ctl->sfull, 1);
        mbar_init(&ctl->sfree, kMath / 32);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&ctl->ops_ready[x], kMath / 64);   // the eight warps of a column half
            mbar_init(&ctl->d_done[x], 1);
            mbar_init(&ctl->aready[x], kMath / 32);      // all sixteen math warps
            mbar_init(&ctl->afree[x], 2);                // both issuers
        }
        ctl->abort = 0;
        mbar_fence_init();
        tma_prefetch(&tm_m);
        tma_prefetch(&tm_s);
        if (a.S_init) tma_prefetch(&tm_i);
        tma_prefetch(&tm_o);
    }
    if (warp == 1) tmem_alloc(&ctl->tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;

    if (warp == 0) {
        // ------------------------------------------------------------ producers: M_p and S_init (lane 0), S_p (lane 1)
        if (lane == 0) {
            // fills of the M_p stage, in the order the math warps take them: the first
            // unit's S_init, then per unit its M_p in step order with the unit's S_init
            // after its first M_p (for the first unit: before it)
            uint32_t f = 0;
            bool first = true;
            auto fill = [&](const CUtensorMap *tm, int row) -> bool {
                if (f >= 1 && !mbar_wait(&ctl->mfree, (f - 1) & 1u)) *abortp = 1;
                if (*abortp) return false;
                mbar_expect_tx(&ctl->mfull, 65536u);
#pragma unroll
                for (int bx = 0; bx < 4; ++bx)
                    tma_load_3d(smem + kMstage + bx * 16384, tm, &ctl->mfull, 32 * bx, 0, row);
                ++f;
                return true;
            };
            for (int64_t u = blockIdx.x; u < units && !*abortp; u += gridDim.x) {
                const int n = unit_steps(a, u, true);
                if (n == 0) continue;   // the math warps copy S_init over
                if (first && a.S_init && !fill(&tm_i, (int)(u * kD))) break;
                for (int c = 0; c < n; ++c) {
                    if (!fill(&tm_m, (int)(step_entry(a, u, c, true) * kD))) break;
                    if (c == 0 && !first && a.S_init && !fill(&tm_i, (int)(u * kD))) break;
                }
                first = false;
            }
            if (*abortp && f > 0) mbar_wait(&ctl->mfull, (f - 1) & 1u);   // the last copy lands
        } else if (lane == 1 && !OP) {   // (operator mode reads no S_p)
            int64_t g = 0;   // steps of this CTA so far
            for (int64_t u = blockIdx.x; u < units && !*abortp; u += gridDim.x) {
                const int n = unit_steps(a, u, false);
                for (int c = 0; c < n; ++c, ++g) {
                    // the stage's previous step is done with (S_p read, a result stored from it)
                    if (g >= 1 && !mbar_wait(&ctl->sfree, (uint32_t)(g - 1) & 1u)) *abortp = 1;
                    if (*abortp) break;
                    const int row = (int)(step_entry(a, u, c, false) * kD);
                    mbar_expect_tx(&ctl->sfull, 65536u);
#pragma unroll
                    for (int bx = 0; bx < 4; ++bx)
                        tma_load_3d(smem + kSstage + bx * 16384, &tm_s, &ctl->sfull, 32 * bx, 0, row);
                }
            }
            if (*abortp && g > 0) mbar_wait(&ctl->sfull, (uint32_t)(g - 1) & 1u);   // the last copy lands
        }
    } else if (warp == 1 || warp == 18) {
        // ------------------------------------------------------------ MMA issuers: warp 1 takes
        // columns 0..63 of D, warp 18 columns 64..127 (N = 64 products from two threads issue
        // at nearly twice the rate of N = 128 products from one)
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 64, false, true);   // A TMEM, B MN-major
            const uint32_t nh = warp == 1 ? 0u : 1u;
            const uint32_t b0 = smem_addr(smem) + nh * 16384u;   // the B atom of this column half
            const uint32_t dcol = tmem + kTd + nh * 64u;
            // B descriptors of the three parts, built once: a k step of 16 rows (2048 bytes)
            // adds 2048 >> 4 to the start-address field
            const uint64_t dh0 = smem_desc_sw128(b0, 16384, 1024);
            const uint64_t dm0 = smem_desc_sw128(b0 + kBpart, 16384, 1024);
            const uint64_t dl0 = smem_desc_sw128(b0 + 2 * kBpart, 16384, 1024);
            int64_t g = 0;
            for (int64_t u = blockIdx.x; u < units && !*abortp; u += gridDim.x) {
                const int n = unit_steps(a, u, false);
                for (int c = 0; c < n; ++c, ++g) {
                    // this half's B and the step's A operand are in place
                    if (!mbar_wait(&ctl->ops_ready[nh], (uint32_t)g & 1u) ||
                        !mbar_wait(&ctl->aready[g & 1], (uint32_t)(g >> 1) & 1u) || *abortp) {
                        *abortp = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t abuf = tmem + kTa + (uint32_t)(g & 1) * 192u;
                    if (NS == 2) {
                        // hi / lo parts (at the mid positions): lo products first, then hi x hi
#pragma unroll 4
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint32_t off = (uint32_t)ks * 2048u;
                            const uint64_t bh = dh0 + (uint64_t)(ks * 128);
                            const uint64_t bl = dm0 + (uint64_t)(ks * 128);
                            const uint32_t ah = abuf + (uint32_t)ks * 8u, al = ah + 64u;
                            mma_f16_ta(dcol, ah, bl, idesc, ks > 0);
                            mma_f16_ta(dcol, al, bh, idesc, 1u);
                        }
#pragma unroll 4
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint64_t bh = dh0 + (uint64_t)(ks * 128);
                            mma_f16_ta(dcol, abuf + (uint32_t)ks * 8u, bh, idesc, 1u);
                        }
                    } else if (OP) {
                        // operator chains: smallest terms first.  The unit rounds each
                        // instruction's sum into the fp32 accumulator; nothing decays an
                        // operator chain's early error, so the 2^-16-level products (hl, mm,
                        // lh) and then the 2^-8-level ones (hm, mh) are summed while the
                        // accumulator is still small and only the eight hi x hi products
                        // round at full magnitude
#pragma unroll 2
                        for (int ks = 0; ks < 8; ++ks) {   // K = 128 in steps of 16 (two 8-row groups of B)
                            const uint32_t off = (uint32_t)ks * 2048u;
                            const uint64_t bh = dh0 + (uint64_t)(ks * 128);
                            const uint64_t bm = dm0 + (uint64_t)(ks * 128);
                            const uint64_t bl = dl0 + (uint64_t)(ks * 128);
                            const uint32_t ah = abuf + (uint32_t)ks * 8u, am = ah + 64u, al = ah + 128u;
                            mma_f16_ta(dcol, ah, bl, idesc, ks > 0);
                            mma_f16_ta(dcol, am, bm, idesc, 1u);
                            mma_f16_ta(dcol, al, bh, idesc, 1u);
                        }
#pragma unroll 2
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint32_t off = (uint32_t)ks * 2048u;
                            const uint64_t bh = dh0 + (uint64_t)(ks * 128);
                            const uint64_t bm = dm0 + (uint64_t)(ks * 128);
                            const uint32_t ah = abuf + (uint32_t)ks * 8u, am = ah + 64u;
                            mma_f16_ta(dcol, ah, bm, idesc, 1u);
                            mma_f16_ta(dcol, am, bh, idesc, 1u);
                        }
#pragma unroll 4
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint64_t bh = dh0 + (uint64_t)(ks * 128);
                            mma_f16_ta(dcol, abuf + (uint32_t)ks * 8u, bh, idesc, 1u);
                        }
                    } else {
                        // state chains (each step decays the earlier error): per k-step
#pragma unroll 2
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint32_t off = (uint32_t)ks * 2048u;
                            const uint64_t bh = dh0 + (uint64_t)(ks * 128);
                            const uint64_t bm = dm0 + (uint64_t)(ks * 128);
                            const uint64_t bl = dl0 + (uint64_t)(ks * 128);
                            const uint32_t ah = abuf + (uint32_t)ks * 8u, am = ah + 64u, al = ah + 128u;
                            mma_f16_ta(dcol, ah, bh, idesc, ks > 0);
                            mma_f16_ta(dcol, ah, bm, idesc, 1u);
                            mma_f16_ta(dcol, am, bh, idesc, 1u);
                            mma_f16_ta(dcol, ah, bl, idesc, 1u);
                            mma_f16_ta(dcol, am, bm, idesc, 1u);
                            mma_f16_ta(dcol, al, bh, idesc, 1u);
                        }
                    }
                    mma_commit(&ctl->d_done[nh]);
                    mma_commit(&ctl->afree[g & 1]);
                }
            }
            if (*abortp) {   // drain: completes once every MMA this thread issued is done
                mma_commit(&ctl->d_done[nh]);
                mbar_wait(&ctl->d_done[nh], (uint32_t)g & 1u);
            }
        }
    } else {
        // ------------------------------------------------------------ math warps
        const int cq = (warp - 2) >> 2;              // column quarter: [32 cq, 32 cq + 32)
        const int hh = cq >> 1;                      // column half: its own pipeline
        const int hbar = 2 + hh;                     // named barrier of the half's 256 threads
        const int quarter = warp & 3;
        const int i = quarter * 32 + lane;           // row of S / of M_p
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int64_t DD = (int64_t)kD * kD;
        float srow[32];                              // exact running state, row i, 32 columns
        uint32_t f = 0;                              // fills of the M_p stage taken (parity)

        // split M_p of step g (the stage's next fill) into TMEM operand buffer g & 1, once
        // both halves' products of step g - 2 are done with that buffer
        auto split_m = [&](int64_t g) -> bool {
            if (!bar_and(hbar, kMath / 2,
                         (g < 2 || mbar_wait(&ctl->afree[g & 1], (uint32_t)((g - 2) >> 1) & 1u)) &&
                             mbar_wait(&ctl->mfull, f & 1u) && !*abortp))
                return false;
            tc_fence_after();
            const uint8_t *ms = smem + kMstage;
            uint32_t hi[16], mid[16], lo[16];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int col = cq * 32 + 4 * q;
                const int box = col >> 5, chunk = (col & 31) >> 2;
                const float4 m4 =
                    *reinterpret_cast<const float4 *>(ms + box * 16384 + i * 128 + ((chunk ^ (i & 7)) << 4));
                if (NS == 3) {
                    split3_pair(m4.x, m4.y, hi[2 * q], mid[2 * q], lo[2 * q]);
                    split3_pair(m4.z, m4.w, hi[2 * q + 1], mid[2 * q + 1], lo[2 * q + 1]);
                } else {   // hi / lo: the second part goes where mid goes
                    split2_pair(m4.x, m4.y, hi[2 * q], mid[2 * q]);
                    split2_pair(m4.z, m4.w, hi[2 * q + 1], mid[2 * q + 1]);
                }
            }
            const uint32_t ab = tmem + lane_off + kTa + (uint32_t)(g & 1) * 192u + (uint32_t)(cq * 16);
            tmem_st16(ab, hi);
            tmem_st16(ab + 64u, mid);
            if (NS == 3) tmem_st16(ab + 128u, lo);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ctl->mfree);            // the stage may take its next fill
                mbar_arrive(&ctl->aready[g & 1]);    // this warp's share of the A operand is in
            }
            ++f;
            return true;
        };
        // a unit without steps: S_out = S_init (or 0; operator mode: I)
        auto copy_init = [&](int64_t u) {
            const float4 *init =
                a.S_init ? reinterpret_cast<const float4 *>(a.S_init + u * DD + i * kD + cq * 32) : nullptr;
            float4 *out = reinterpret_cast<float4 *>(a.S_out + u * DD + i * kD + cq * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (OP) {
                    const int c0 = cq * 32 + 4 * q;
                    out[q] = make_float4(i == c0 ? 1.f : 0.f, i == c0 + 1 ? 1.f : 0.f, i == c0 + 2 ? 1.f : 0.f,
                                         i == c0 + 3 ? 1.f : 0.f);
                } else {
                    out[q] = init ? init[q] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            if (OP && threadIdx.x == 64) a.lam_out[u] = 0.f;
        };

        auto load_init = [&]() -> bool {   // S_init row of the next unit (the stage's next fill, or 0) into srow
            if (!a.S_init) {   // zero, or the identity in operator mode
#pragma unroll
                for (int q = 0; q < 32; ++q) srow[q] = (OP && i == cq * 32 + q) ? 1.f : 0.f;
                return true;
            }
            if (!bar_and(hbar, kMath / 2, mbar_wait(&ctl->mfull, f & 1u) && !*abortp)) return false;
            const uint8_t *ms = smem + kMstage + cq * 16384 + i * 128;   // box cq: this thread's 32 columns
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(ms + ((q ^ (i & 7)) << 4));
                srow[4 * q] = v.x; srow[4 * q + 1] = v.y; srow[4 * q + 2] = v.z; srow[4 * q + 3] = v.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->mfree);
            ++f;
            return true;
        };
        // the next unit of this CTA after uu that has steps (units without steps are written here)
        auto next_unit = [&](int64_t uu) {
            uu += gridDim.x;
            while (uu < units && unit_steps(a, uu, false) == 0) {
                copy_init(uu);
                uu += gridDim.x;
            }
            return uu;
        };

        int64_t g = 0;
        bool ok = true;
        int op_exp = 0;     // operator mode: power of two taken out of the unit's product so far
        uint32_t nrn = 0;   // operator mode: renormalisations so far (parity of the maxima buffer)
        int64_t u = next_unit((int64_t)blockIdx.x - gridDim.x);
        if (u < units) ok = load_init() && split_m(0);   // the first unit's state, its first step's operand
        while (ok && u < units) {
            const int n = unit_steps(a, u, false);
            const int64_t un = next_unit(u);
            for (int c = 0; c < n && ok; ++c, ++g) {
                const bool last = c + 1 == n;
                const int64_t e = step_entry(a, u, c, false);
                // B = S (bf16 hi / mid / lo) -> shared memory, MN-major: row k = i, n contiguous,
                // 2 atoms of 64 columns, 128-byte swizzle.  B is free: the last products are done.
#pragma unroll
                for (int q = 0; q < 4; ++q) {              // 8 columns (one 16-byte chunk) at a time
                    const int chunk = (cq & 1) * 4 + q;
                    const int off = (cq >> 1) * 16384 + i * 128 + ((chunk ^ (i & 7)) << 4);
                    uint32_t h[4], md[4], l[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        if (NS == 3) split3_pair(srow[8 * q + 2 * p], srow[8 * q + 2 * p + 1], h[p], md[p], l[p]);
                        else split2_pair(srow[8 * q + 2 * p], srow[8 * q + 2 * p + 1], h[p], md[p]);
                    }
                    *reinterpret_cast<uint4 *>(smem + off) = make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4 *>(smem + kBpart + off) = make_uint4(md[0], md[1], md[2], md[3]);
                    if (NS == 3)
                        *reinterpret_cast<uint4 *>(smem + 2 * kBpart + off) = make_uint4(l[0], l[1], l[2], l[3]);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->ops_ready[hh]);
                // while the products run: the next step's M_p into the other operand buffer
                if ((!last || un < units) && !split_m(g + 1)) {
                    ok = false;
                    break;
                }
                const float scale = OP ? 1.f : expf(a.pool_lam[e]);
                if (!bar_and(hbar, kMath / 2,
                             (OP || mbar_wait(&ctl->sfull, (uint32_t)g & 1u)) &&
                                 mbar_wait(&ctl->d_done[hh], (uint32_t)g & 1u) && !*abortp)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // S <- scale D + S_p (S_p from the stage: box cq holds this thread's 32 columns),
                // 16 columns at a time
                uint8_t *sp = smem + kSstage + cq * 16384 + i * 128;
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    uint32_t dv[16];
                    tmem_ld16(tmem + lane_off + kTd + (uint32_t)(cq * 32 + hb * 16), dv);
                    tmem_wait_ld();
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int q = hb * 4 + q4;
                        const float4 v = OP ? make_float4(0.f, 0.f, 0.f, 0.f)
                                              : *reinterpret_cast<const float4 *>(sp + ((q ^ (i & 7)) << 4));
                        const uint64_t sc2 = pk2(scale, scale);
                        float4 r;
                        upk2(fma2(sc2, pk2(__uint_as_float(dv[4 * q4]), __uint_as_float(dv[4 * q4 + 1])),
                                  pk2(v.x, v.y)),
                             r.x, r.y);
                        upk2(fma2(sc2, pk2(__uint_as_float(dv[4 * q4 + 2]), __uint_as_float(dv[4 * q4 + 3])),
                                  pk2(v.z, v.w)),
                             r.z, r.w);
                        if (last) {   // in place: the stage then leaves by TMA store
                            *reinterpret_cast<float4 *>(sp + ((q ^ (i & 7)) << 4)) = r;
                        } else {
                            srow[4 * q] = r.x; srow[4 * q + 1] = r.y; srow[4 * q + 2] = r.z; srow[4 * q + 3] = r.w;
                        }
                    }
                }
                tc_fence_before();
                if (OP && !last && (c & 3) == 3) {
                    // operator mode: bring max|M| back to [1, 2) by a power of two every 4 steps
                    // (all sixteen warps agree on it: the scaling must be one for the matrix)
                    float mx = 0.f;
#pragma unroll
                    for (int q = 0; q < 32; ++q) mx = fmaxf(mx, fabsf(srow[q]));
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    float *rm = ctl->rmax[nrn & 1];
                    if (lane == 0) rm[warp - 2] = mx;
                    bar_sync(1, kMath);
                    mx = 0.f;
#pragma unroll
                    for (int x = 0; x < 16; ++x) mx = fmaxf(mx, rm[x]);
                    ++nrn;
                    if (mx > 0.f && (mx < 1.f || mx >= 2.f)) {
                        int ex;
                        frexpf(mx, &ex);
                        const float sc = ldexpf(1.f, 1 - ex);
#pragma unroll
                        for (int q = 0; q < 32; ++q) srow[q] *= sc;
                        op_exp += ex - 1;
                    }
                }
                if (last) {
                    fence_async_smem();    // the results, visible to the TMA store
                    bar_sync(hbar, kMath / 2);
                    if (threadIdx.x == 64 + hh * 256) {   // each half stores its two boxes
#pragma unroll
                        for (int bx = 2 * hh; bx < 2 * hh + 2; ++bx)
                            tma_store_3d(&tm_o, smem + kSstage + bx * 16384, 32 * bx, 0, (int)(u * kD));
                        bulk_commit();
                        bulk_wait_read_all();   // the stage is read: it may take the next S_p
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->sfree);   // the stage may take the next step's S_p
                if (OP && last) {   // the unit's exponent, then a fresh one for the next
                    if (threadIdx.x == 64) a.lam_out[u] = (float)op_exp;
                    op_exp = 0;
                }
                // after a unit's last step: the next unit's S_init (its fill has been in flight
                // since the next unit's first M_p was split)
                if (last && un < units && !load_init()) {
                    ok = false;
                    break;
                }
            }
            u = un;
        }
        if (!ok) *abortp = 1;
        if (threadIdx.x == 64 || threadIdx.x == 320) bulk_wait_all();   // the stores of S_out are complete
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abortp && a.d_err) atomicExch(a.d_err, (int)HYPIC_ETIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool chain_dense_tc_supported(const ChainArgs &a) {
    const int64_t units = (int64_t)a.R * a.n_layers * a.H;
    return a.fam == HYPIC_DENSE && a.dk == 128 && a.dv == 128 && a.P > 0 &&
           (int64_t)a.P * a.n_layers * a.H * 128 < ((int64_t)1 << 31) && units * 128 < ((int64_t)1 << 31) &&
           tensor_map_encoder() != nullptr;
}

cudaError_t launch_chain_dense_tc(const ChainArgs &a, cudaStream_t s) {
    const int64_t units = (int64_t)a.R * a.n_layers * a.H;
    if (units == 0) return cudaSuccess;
    CUtensorMap tm, ts, ti, to;
    const uint64_t rows = (uint64_t)a.P * a.n_layers * a.H * 128, urows = (uint64_t)units * 128;
    if (!make_tensor_map_3d(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.pool_M, 128, 1, rows, 32, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.pool_S, 128, 1, rows, 32, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&to, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.S_out, 128, 1, urows, 32, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    ti = to;   // unused without S_init
    if (a.S_init && !make_tensor_map_3d(&ti, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.S_init, 128, 1, urows, 32, 128,
                                        CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    auto kern = a.two_way ? (a.op ? chain_dense_tc_kernel<true, 2> : chain_dense_tc_kernel<false, 2>)
                          : (a.op ? chain_dense_tc_kernel<true, 3> : chain_dense_tc_kernel<false, 3>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t grid = units < sms ? units : sms;   // persistent: one CTA per SM
    kern<<<(unsigned)grid, kThreads, kSmem, s>>>(tm, ts, ti, to, a, units);
    return cudaGetLastError();
}

}  // namespace hypic
