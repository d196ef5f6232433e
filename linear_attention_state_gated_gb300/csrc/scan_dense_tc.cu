// scan_dense_tc.cu -- gated delta rule segment scan on tcgen05 tensor cores.
//
// Chunked WY/UT form of S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
// (C = 64 tokens per chunk; b_t = in-chunk cumulative decay, b_C its total):
//   L_ts = beta_t (b_t / b_s) k_t.k_s  (s < t),   A = (I + L)^-1
//   for X = [M | S] (the transition and the state side by side, d x 2d):
//   P = K X_0,  R = diag(beta) [0 | V] - diag(beta b) P,  Delta = A R,
//   X <- b_C X_0 + K^T diag(b_C / b) Delta.
// Within a chunk delta_t = beta_t (v_t - alpha_t S_{t-1}^T k_t) satisfies
// (I + L) Delta = R, which is where the triangular system comes from.
//
// Every product above acts on one column of X at a time, so the transition
// half M and the state half S of a chain are handled by two CTAs (launched
// side by side).  A CTA keeps its half transposed in TMEM (column m of X on
// TMEM lane m, key channel k along the columns), so every product is M = 128:
//   Gram   G   = K K^T                  (bf16 keys, exact products)
//   P^T        = X0^T K^T               (X0 split into bf16 hi + lo, from TMEM)
//   Delta^T    = R^T A^T                (3-term bf16 split of both operands)
//   X^T       += (Delta~)^T K           (Delta~ split hi + lo, K exact)
// X0, R and Delta~ never leave TMEM (the state warps convert them in place
// with tcgen05.ld / st); A goes through shared memory.  The transition half is
// rescaled by a power of two every chunk (exponent into lambda), so
// T_C = exp(lambda) M with max|M| in [1, 2) at the end.
//
// Warp roles: 0 TMA; 1 MMA issue; 2-9 "prep" (gates, Gram -> L -> blocked
// (I+L)^-1 -> A operand), which depends only on the chunk's keys and gates and
// runs one chunk ahead; 10-17 "state" (TMEM round trip of X, R, Delta~,
// epilogue).  Every wait is time-bounded; a timeout is reported as
// HYPIC_ETIMEOUT.
#include "internal.cuh"
#include "dense_common.cuh"
#include "sm100.cuh"

namespace hypic {
namespace {

using namespace sm100;
using dense::split_pair;
using dense::wait_or_abort;
using dense::exponent_of;

constexpr int kC = dense::kC;    // tokens per chunk
constexpr int kD = 128;         // d_k = d_v
constexpr int kNS = 2;          // TMA stages
constexpr int kThreads = 576;   // 18 warps
constexpr int kPrep = 256;      // warps 2..9
constexpr int kState = 256;     // warps 10..17
constexpr int kLd = dense::kLd;  // padded row stride of the fp32 L / A work tiles

// shared memory map (offsets from the 1024-aligned base)
constexpr int kBox = kC * 128;              // 64 channels x 64 tokens, bf16: 8 KB
constexpr int kTile = 2 * kBox;             // 128 channels: 16 KB
constexpr int kStage = 2 * kTile;           // K tile, V tile
constexpr int kAop = kNS * kStage;          // A operands, two buffers x (hi, lo) (8 KB each)
constexpr int kLws = kAop + 4 * 8192;       // fp32 L (64 x 65)
constexpr int kAws = kLws + kC * kLd * 4;   // fp32 A (64 x 65)
constexpr int kTws = kAws + kC * kLd * 4;   // fp32 temporaries for the off-diagonal blocks (3 x 16 x 16)
constexpr int kCtl = kTws + 3 * 256 * 4;

// TMEM column map (512 columns allocated)
constexpr uint32_t kTx = 0;       // X^T half, fp32 (128 columns)
constexpr uint32_t kTxop = 128;   // X0^T operand: hi [128, 192), lo [192, 256), bf16 pairs
constexpr uint32_t kTacc = 256;   // P^T / Delta^T accumulator (64 columns)
constexpr uint32_t kTopr = 320;   // R^T / Delta~^T operand: hi [320, 352), lo [352, 384)
constexpr uint32_t kTgram = 384;  // Gram (64 columns)

struct DenseCtrl {
    uint64_t full[kNS], empty[kNS];
    uint64_t gram_done, gfree, p_done, d_done, x_done;
    uint64_t ops_ready, r_ready, dt_ready;
    uint64_t gates_ready[2], aop_ready[2], aop_free[2];
    float gl[2][kC], gbb[2][kC], gw[2][kC], gbeta[2][kC];   // per chunk parity: Lambda_t, beta_t b_t,
    float bC[2];                                             // b_C / b_t, beta_t; b_C
    float redmax[8];
    uint32_t tmem;
    int abort;
};

constexpr int kSmem = kCtl + (int)sizeof(DenseCtrl) + 1024;
static_assert(kSmem <= 232448, "fits in one SM's shared memory");

// max over the 8 state warps (named barrier 2)
__device__ __forceinline__ float state_max(float mx, DenseCtrl *ctl, int sw, int lane) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) ctl->redmax[sw] = mx;
    bar_sync(2, kState);
    mx = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) mx = fmaxf(mx, ctl->redmax[w]);
    bar_sync(2, kState);
    return mx;
}

__global__ void __launch_bounds__(kThreads, 1)   // 18 warps: <= 96 registers per thread
    scan_dense_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const ScanArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    DenseCtrl *ctl = reinterpret_cast<DenseCtrl *>(smem + kCtl);
    volatile int *abortp = &ctl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int half = blockIdx.x & 1;   // 0: transition M, 1: state S
    const int unit = blockIdx.x >> 1;
    const int h = unit % a.H;
    const int seg = (unit / a.H) % a.n_seg;
    const int l = unit / (a.H * a.n_seg);
    int64_t t0 = a.seg_offsets[seg], t1 = a.seg_offsets[seg + 1];
    const bool bad = !(t0 >= 0 && t0 <= t1 && t1 <= a.N);
    if (bad) t0 = t1 = 0;
    const int nc = (int)((t1 - t0 + kC - 1) / kC);
    const int64_t row0 = (int64_t)l * a.N + t0;   // token row of the segment's first token

    if (threadIdx.x == 0) {
        if (bad) flag_index_error(a.d_err);
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->gram_done, 1);
        mbar_init(&ctl->gfree, 4);
        mbar_init(&ctl->p_done, 1);
        mbar_init(&ctl->d_done, 1);
        mbar_init(&ctl->x_done, 1);
        mbar_init(&ctl->ops_ready, kState / 32);
        mbar_init(&ctl->r_ready, kState / 32);
        mbar_init(&ctl->dt_ready, kState / 32);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->gates_ready[b], 1);
            mbar_init(&ctl->aop_ready[b], kPrep / 32);
            mbar_init(&ctl->aop_free[b], 1);
        }
        ctl->abort = 0;
        mbar_fence_init();
        tma_prefetch(&tm_k);
        if (half) tma_prefetch(&tm_v);
    }
    if (warp == 1) tmem_alloc(&ctl->tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            for (int j = 0; j < nc; ++j) {
                const int s = j % kNS;
                if (!wait_or_abort(&ctl->empty[s], ((uint32_t)(j / kNS) & 1u) ^ 1u, abortp)) break;
                uint8_t *st = smem + s * kStage;
                const int row = (int)(row0 + (int64_t)j * kC);
                mbar_expect_tx(&ctl->full[s], (uint32_t)(half ? 2 * kTile : kTile));
                tma_load_3d(st, &tm_k, &ctl->full[s], 0, h, row);
                tma_load_3d(st + kBox, &tm_k, &ctl->full[s], 64, h, row);
                if (half) {   // V only feeds the state half
                    tma_load_3d(st + kTile, &tm_v, &ctl->full[s], 0, h, row);
                    tma_load_3d(st + kTile + kBox, &tm_v, &ctl->full[s], 64, h, row);
                }
                issued = j + 1;
            }
            if (*abortp)
                for (int j = issued - kNS < 0 ? 0 : issued - kNS; j < issued; ++j)
                    mbar_wait(&ctl->full[j % kNS], (uint32_t)(j / kNS) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_n64 = idesc_bf16_f32(128, 64, false, false);     // A, B K-major
            constexpr uint32_t id_u = idesc_bf16_f32(128, 128, false, true);       // B = K (MN-major)
            auto gram = [&](int j) {   // G = K K^T (M padded to 128 rows; rows >= 64 unused)
                const uint32_t kb = smem_addr(smem + (j % kNS) * kStage);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (uint32_t)(ks >> 2) * kBox + (uint32_t)(ks & 3) * 32u;
                    mma_f16(tmem + kTgram, smem_desc_sw128(kb + off, 0, 1024), smem_desc_sw128(kb + off, 0, 1024),
                            id_n64, ks > 0);
                }
                mma_commit(&ctl->gram_done);
            };
            bool run = nc > 0 && wait_or_abort(&ctl->full[0], 0, abortp);
            if (run) {
                tc_fence_after();
                gram(0);
            }
            for (int j = 0; run && j < nc; ++j) {
                const int s = j % kNS;
                const uint32_t par = (uint32_t)j & 1u;
                const uint32_t kb = smem_addr(smem + s * kStage);
                // P^T = X0^T K^T, X0 as hi + lo
                if (!wait_or_abort(&ctl->ops_ready, par, abortp)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kk = (uint32_t)(ks >> 2) * kBox + (uint32_t)(ks & 3) * 32u;
                    const uint64_t bd = smem_desc_sw128(kb + kk, 0, 1024);
                    mma_f16_ta(tmem + kTacc, tmem + kTxop + (uint32_t)ks * 8u, bd, id_n64, ks > 0);
                    mma_f16_ta(tmem + kTacc, tmem + kTxop + 64u + (uint32_t)ks * 8u, bd, id_n64, 1u);
                }
                mma_commit(&ctl->p_done);
                // next chunk's Gram as soon as its keys are in and the prep warps read this one
                if (j + 1 < nc) {
                    if (!wait_or_abort(&ctl->full[(j + 1) % kNS], (uint32_t)((j + 1) / kNS) & 1u, abortp) ||
                        !wait_or_abort(&ctl->gfree, par, abortp))
                        break;
                    tc_fence_after();
                    gram(j + 1);
                }
                // Delta^T = R^T A^T, three-term split
                if (!wait_or_abort(&ctl->r_ready, par, abortp) ||
                    !wait_or_abort(&ctl->aop_ready[par], (uint32_t)(j >> 1) & 1u, abortp))
                    break;
                tc_fence_after();
                const uint32_t aop = smem_addr(smem + kAop + (int)par * 16384);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t ah = smem_desc_sw128(aop + (uint32_t)ks * 32u, 0, 1024);
                    const uint64_t al = smem_desc_sw128(aop + 8192u + (uint32_t)ks * 32u, 0, 1024);
                    const uint32_t c = (uint32_t)ks * 8u;
                    mma_f16_ta(tmem + kTacc, tmem + kTopr + c, ah, id_n64, ks > 0);
                    mma_f16_ta(tmem + kTacc, tmem + kTopr + c, al, id_n64, 1u);
                    mma_f16_ta(tmem + kTacc, tmem + kTopr + 32u + c, ah, id_n64, 1u);
                }
                mma_commit(&ctl->d_done);
                mma_commit(&ctl->aop_free[par]);
                // X^T += Delta~^T K (K as the MN-major B operand: row t, channels contiguous)
                if (!wait_or_abort(&ctl->dt_ready, par, abortp)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t bd = smem_desc_sw128(kb + (uint32_t)ks * 2048u, kBox, 1024);
                    const uint32_t c = (uint32_t)ks * 8u;
                    mma_f16_ta(tmem + kTx, tmem + kTopr + c, bd, id_u, 1u);
                    mma_f16_ta(tmem + kTx, tmem + kTopr + 32u + c, bd, id_u, 1u);
                }
                mma_commit(&ctl->x_done);
                mma_commit(&ctl->empty[s]);
            }
            if (*abortp) {
                mma_commit(&ctl->p_done);   // drain: completes once issued MMAs are done
                mbar_wait(&ctl->p_done, nc & 1);
            }
        }
    } else if (warp < 10) {
        // ------------------------------------------------------------ prep warps
        const int pt = threadIdx.x - 64;            // 0..255
        const int quarter = warp & 3;
        const int gcol = (warp - 2) >> 2;           // Gram column half this warp reads
        float *Lw = reinterpret_cast<float *>(smem + kLws);
        float *Aw = reinterpret_cast<float *>(smem + kAws);
        float *Tw = reinterpret_cast<float *>(smem + kTws);
        float pa[2], pb[2];
        auto prefetch = [&](int j) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int64_t t = t0 + (int64_t)j * kC + lane + 32 * q;
                const bool v = j < nc && t < t1;
                const int64_t row = ((int64_t)l * a.N + t) * a.H + h;
                pa[q] = v ? a.alpha[row] : 1.f;
                pb[q] = v ? (a.beta ? a.beta[row] : 1.f) : 0.f;
            }
        };
        if (warp == 2) prefetch(0);
        for (int j = 0; j < nc; ++j) {
            const uint32_t par = (uint32_t)j & 1u;
            if (!bar_and(1, kPrep, mbar_wait(&ctl->gram_done, par) && !*abortp)) {
                *abortp = 1;
                break;
            }
            // ---- gates: Lambda (inclusive in-chunk log decay), beta b, b_C / b.  Written only
            // after Gram(j) exists: the state warps are then done with chunk j-2 (same buffer).
            if (warp == 2) {
                float lg[2], inc[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) lg[q] = logf(pa[q]);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float x = lg[q];
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, x, off);
                        if (lane >= off) x += y;
                    }
                    inc[q] = x;
                }
                const float tot0 = __shfl_sync(0xffffffffu, inc[0], 31);
                inc[1] += tot0;
                const float total = __shfl_sync(0xffffffffu, inc[1], 31);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int t = lane + 32 * q;
                    ctl->gl[par][t] = inc[q];
                    ctl->gbb[par][t] = pb[q] * expf(inc[q]);
                    ctl->gw[par][t] = expf(total - inc[q]);
                    ctl->gbeta[par][t] = pb[q];
                }
                if (lane == 0) ctl->bC[par] = expf(total);
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->gates_ready[par]);
                if (j + 1 < nc) prefetch(j + 1);
            }
            bar_sync(1, kPrep);
            tc_fence_after();
            // ---- L[t][s] = beta_t exp(Lambda_t - Lambda_s) G[t][s] for s < t (rows t < 64)
            if (quarter < 2) {
                const int t = quarter * 32 + lane;   // 0..63
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + kTgram + (uint32_t)(gcol * 32), r);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->gfree);   // the Gram columns may be overwritten
                const float lt = ctl->gl[par][t], bt = ctl->gbeta[par][t];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int sc = gcol * 32 + i;
                    Lw[t * kLd + sc] = sc < t ? bt * __expf(lt - ctl->gl[par][sc]) * __uint_as_float(r[i]) : 0.f;
                }
            }
            bar_sync(1, kPrep);
            // ---- A = (I + L)^-1 (blocked, shared memory)
            dense::tri_inverse<kPrep, 1>(Lw, Aw, Tw, pt);
            // ---- A -> bf16 hi / lo operand tiles (row t, s contiguous, 128-byte swizzle)
            if (!bar_and(1, kPrep, mbar_wait(&ctl->aop_free[par], ((uint32_t)(j >> 1) & 1u) ^ 1u) && !*abortp)) {
                *abortp = 1;
                break;
            }
            {
                uint8_t *aop = smem + kAop + (int)par * 16384;
                const int t = pt >> 2, c0 = (pt & 3) * 2;   // two 8-element chunks per thread
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = c0 + cc;
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p)
                        split_pair(Aw[t * kLd + c * 8 + 2 * p], Aw[t * kLd + c * 8 + 2 * p + 1], hi[p], lo[p]);
                    const int off = t * 128 + ((c ^ (t & 7)) << 4);
                    *reinterpret_cast<uint4 *>(aop + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(aop + 8192 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->aop_ready[par]);
            bar_sync(1, kPrep);   // the work tiles are reused by the next chunk
        }
    } else {
        // ------------------------------------------------------------ state warps
        const int st = threadIdx.x - 320;           // 0..255
        const int sw = warp - 10;                   // 0..7
        const int ch = sw >> 2;                     // which half of the columns this warp converts
        const int quarter = warp & 3;               // TMEM lanes this warp may touch
        const int m = quarter * 32 + lane;          // column of X = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tx = tmem + lane_off + kTx + (uint32_t)(ch * 64);
        const uint32_t txop = tmem + lane_off + kTxop + (uint32_t)(ch * 32);
        const uint32_t tacc = tmem + lane_off + kTacc + (uint32_t)(ch * 32);
        const uint32_t topr = tmem + lane_off + kTopr + (uint32_t)(ch * 16);
        // Transition half: M_true = exp(lam_d + lam_exp ln2) M_stored, and each chunk
        // stores T_chunk M / b_C (log b_C into lam_d).  State half: S_true =
        // exp(ls) S_stored.  Either way the update only accumulates into TMEM; X is
        // rewritten only to renormalise (every 8 chunks for M, when ls < -20 for S)
        // or on a chunk whose total decay exceeds e^-40 (exact write-back form).
        int lam_exp = 0;
        double lam_d = 0.0;
        float ls = 0.f;

        // initial X^T: identity (transition) or zero (state)
        {
            uint32_t r[32];
            for (int cb = 0; cb < 2; ++cb) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    r[i] = __float_as_uint((half == 0 && ch * 64 + cb * 32 + i == m) ? 1.f : 0.f);
                tmem_st32(tx + (uint32_t)(cb * 32), r);
            }
            tmem_wait_st();
        }

        for (int j = 0; j < nc; ++j) {
            const int s = j % kNS;
            const uint32_t par = (uint32_t)j & 1u;
            // ---- X round trip (TMEM only): operand X0 (scaled, hi + lo), X <- b_C X0 (scaled)
            bool ok = mbar_wait(&ctl->gates_ready[par], (uint32_t)(j >> 1) & 1u);
            if (j > 0) ok = ok && mbar_wait(&ctl->x_done, par ^ 1u);
            if (!bar_and(2, kState, ok && !*abortp)) {
                *abortp = 1;
                break;
            }
            tc_fence_after();
            const float LC = ctl->gl[par][kC - 1];      // log of the chunk's total decay
            const bool slow = LC < -40.f;
            const bool renorm = slow || (half == 0 ? (j % 8 == 0) : (ls < -20.f));
            float g = 1.f;        // operand = g * X_stored
            float wscale = 1.f;   // X_stored <- g * wscale * X_stored when rewritten
            float fP, fD;         // multipliers of beta*b (in R) and b_C / b (in Delta~)
            if (half == 0) {
                if (renorm) {
                    float mx = 0.f;
                    for (int cb = 0; cb < 2; ++cb) {
                        uint32_t r[32];
                        tmem_ld32(tx + (uint32_t)(cb * 32), r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(__uint_as_float(r[i])));
                    }
                    const int e = exponent_of(state_max(mx, ctl, sw, lane));
                    g = ldexpf(1.f, -e);
                    lam_exp += e;
                }
                wscale = slow ? ctl->bC[par] : 1.f;
                fP = 1.f;
                fD = slow ? 1.f : expf(-LC);
                if (!slow) lam_d += (double)LC;
            } else {
                if (slow) {
                    g = expf(ls);
                    wscale = ctl->bC[par];
                    fP = 1.f;
                    fD = 1.f;
                    ls = 0.f;
                } else {
                    if (renorm) {
                        const int q = (int)rintf(ls * 1.44269504088896341f);
                        g = ldexpf(1.f, q);
                        ls -= (float)q * 0.69314718055994531f;
                    }
                    fP = expf(ls);
                    fD = expf(-(ls + LC));
                    ls += LC;
                }
            }
            const float sc = g * wscale;
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t r[32], hi[16], lo[16];
                tmem_ld32(tx + (uint32_t)(cb * 32), r);
                tmem_wait_ld();
#pragma unroll
                for (int p = 0; p < 16; ++p)
                    split_pair(g * __uint_as_float(r[2 * p]), g * __uint_as_float(r[2 * p + 1]), hi[p], lo[p]);
                tmem_st16(txop + (uint32_t)(cb * 16), hi);
                tmem_st16(txop + 64u + (uint32_t)(cb * 16), lo);
                if (renorm) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(sc * __uint_as_float(r[i]));
                    tmem_st32(tx + (uint32_t)(cb * 32), r);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->ops_ready);
            // ---- R^T = beta [0 | V]^T - (beta b) P^T  -> TMEM operand (hi, lo)
            ok = mbar_wait(&ctl->p_done, par) && mbar_wait(&ctl->full[s], (uint32_t)(j / kNS) & 1u);
            if (!bar_and(2, kState, ok && !*abortp)) {
                *abortp = 1;
                break;
            }
            tc_fence_after();
            {
                const uint8_t *vt = smem + s * kStage + kTile;
                const int vbox = m >> 6, vc = (m & 63) >> 3, vw = (m & 7) * 2;
                uint32_t r[32], hi[16], lo[16];
                tmem_ld32(tacc, r);
                tmem_wait_ld();
#pragma unroll
                for (int p = 0; p < 16; ++p) {
                    float xv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int t = ch * 32 + 2 * p + e;
                        float val = -fP * ctl->gbb[par][t] * __uint_as_float(r[2 * p + e]);
                        if (half) {
                            const uint16_t vb = *reinterpret_cast<const uint16_t *>(
                                vt + vbox * kBox + t * 128 + ((vc ^ (t & 7)) << 4) + vw);
                            val = fmaf(ctl->gbeta[par][t], __uint_as_float((uint32_t)vb << 16), val);
                        }
                        xv[e] = val;
                    }
                    split_pair(xv[0], xv[1], hi[p], lo[p]);
                }
                tmem_st16(topr, hi);
                tmem_st16(topr + 32u, lo);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->r_ready);
            // ---- Delta~^T = Delta^T diag(b_C / b)  -> TMEM operand (hi, lo)
            if (!bar_and(2, kState, mbar_wait(&ctl->d_done, par) && !*abortp)) {
                *abortp = 1;
                break;
            }
            tc_fence_after();
            {
                uint32_t r[32], hi[16], lo[16];
                tmem_ld32(tacc, r);
                tmem_wait_ld();
#pragma unroll
                for (int p = 0; p < 16; ++p) {
                    const int t = ch * 32 + 2 * p;
                    split_pair(fD * ctl->gw[par][t] * __uint_as_float(r[2 * p]),
                               fD * ctl->gw[par][t + 1] * __uint_as_float(r[2 * p + 1]), hi[p], lo[p]);
                }
                tmem_st16(topr, hi);
                tmem_st16(topr + 32u, lo);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->dt_ready);
        }

        // ------------------------------------------------------------ epilogue
        bool ok = true;
        if (nc > 0) ok = mbar_wait(&ctl->x_done, (uint32_t)(nc - 1) & 1u);
        if (bar_and(2, kState, ok && !*abortp)) {
            tc_fence_after();
            const int64_t u_out = ((int64_t)l * a.n_seg + seg) * a.H + h;
            float scale = 1.f;
            if (half == 0) {
                float mx = 0.f;
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(tx + (uint32_t)(cb * 32), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(__uint_as_float(r[i])));
                }
                const int e = exponent_of(state_max(mx, ctl, sw, lane));
                scale = ldexpf(1.f, -e);
                lam_exp += e;
                if (st == 0) a.lam_out[u_out] = (float)(lam_d + (double)lam_exp * 0.69314718055994530942);
            } else {
                scale = expf(ls);
            }
            float *out = (half == 0 ? a.M_out : a.S_out) + u_out * kD * kD;
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t r[32];
                tmem_ld32(tx + (uint32_t)(cb * 32), r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    out[(int64_t)(ch * 64 + cb * 32 + i) * kD + m] = scale * __uint_as_float(r[i]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abortp && a.d_err) atomicExch(a.d_err, (int)HYPIC_ETIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- host side

}  // namespace

bool scan_dense_tc_supported(const ScanArgs &a) {
    return a.fam == HYPIC_DENSE && a.in_dtype == HYPIC_BF16 && a.dk == 128 && a.dv == 128 &&
           a.o_out == nullptr && a.N > 0 && (int64_t)a.n_layers * a.N < ((int64_t)1 << 31) &&
           (int64_t)a.n_layers * a.n_seg * a.H < ((int64_t)1 << 30) &&
           tensor_map_encoder() != nullptr;
}

cudaError_t launch_scan_dense_tc(const ScanArgs &a, cudaStream_t s) {
    const int64_t units = (int64_t)a.n_layers * a.n_seg * a.H;
    if (units == 0) return cudaSuccess;
    const uint64_t rows = (uint64_t)a.n_layers * (uint64_t)a.N;
    CUtensorMap mk, mv;
    if (!make_tensor_map_3d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k, 128, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v, 128, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(scan_dense_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    scan_dense_tc_kernel<<<(unsigned)(2 * units), kThreads, kSmem, s>>>(mk, mv, a);
    return cudaGetLastError();
}

}  // namespace hypic
