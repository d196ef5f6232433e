// scan_sd_o.cu -- scalar-gated segment scan with the per-token outputs o_t on
// tcgen05 tensor cores (RetNet fixed gamma or Mamba2-style per-token decay, optional
// write scale beta), bf16 q / k / v / o, d_k = d_v = 128.
//
// Chunks of C = 64 tokens in order.  With S0 the state at a chunk's start and b_t
// the in-chunk decay (b_t = prod_{r<=t} alpha_r, a scalar per token):
//   o_t = S_t^T q_t = b_t S0^T q_t + sum_{s<=t} (b_t / b_s) beta_s (q_t . k_s) v_s
//       = b_t (O1)_t + (O2)_t,   O1 = Q S0,  O2 = Gq V,
//   Gq[t][s] = [s <= t] (b_t / b_s) beta_s q_t . k_s,
//   S_C = b_C S0 + K~^T V,   K~_s = (b_C / b_s) beta_s k_s.
// The state is kept transposed in TMEM (lane = value channel j, column = key
// channel i), fp32, in its true scale: each chunk's conversion of S0 into the
// bf16 hi / lo operand of O1 also rewrites S <- b_C S0 before the update adds
// K~^T V (every factor above is at most 1, so no scale can overflow; a decay that
// underflows takes S to 0, its limit).  Per CTA one (layer, segment, head):
//   warp 0       TMA: K, V, Q of a chunk (two 64-channel boxes each) into a ring
//                of two stages;
//   warp 1       one thread issues every tcgen05.mma: the Gram G = Q K^T (M = 128,
//                rows 64..127 unused), then per chunk O1^T = S0^T Q^T (S0 split
//                hi + lo), S^T += V^T K~ (K~ split), O2^T = V^T Gq^T (Gq split);
//                lo products first (the unit rounds each instruction's sum into
//                the fp32 accumulator);
//   warps 2-17   gates (log-space prefix sums), Gq and K~ as bf16 hi / lo tiles,
//                the S0 operand, o_t = b_t O1 + O2 (bf16, through a staging tile
//                so that each lane writes 16-byte runs), the final state.
// Every wait is time-bounded; a timeout is reported as HYPIC_ETIMEOUT.
#include "dense_common.cuh"
#include "internal.cuh"
#include "sm100.cuh"

namespace hypic {
namespace {

using namespace sm100;
using dense::split_pair;
using dense::wait_or_abort;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kBox = kC * 128;            // 64 channels x 64 tokens, bf16: 8 KB
constexpr int kNS = 3;                    // TMA stages
constexpr int kCW = 512;                  // conversion threads (16 warps)
constexpr int kThreads = 64 + kCW;

// shared memory, from the 1024-aligned base
constexpr int kStage = 6 * kBox;          // K, V, Q: two boxes each
constexpr int kOffK = 0, kOffV = 2 * kBox, kOffQ = 4 * kBox;
constexpr int kKt = kNS * kStage;         // K~ hi / lo (16 KB each)
constexpr int kGq = kKt + 32768;          // Gq hi / lo (8 KB each), two buffers (chunk parity)
constexpr int kOst = kGq + 2 * 16384;     // o staging: 8 tokens x 32 channels per warp
constexpr int kCtl = kOst + 16 * 512;

struct Ctl {
    uint64_t full[kNS], empty[kNS];
    uint64_t gram_done, gk_ready, xop_ready, x_done, o_done, o_free, drain;
    // gates of a chunk in slot j % 3 (the group's first warp writes chunk j + 1's
    // while other warps may still read chunk j - 1's for its outputs)
    float lt[3][kC];      // in-chunk log decay Lambda_t (inclusive)
    float bt[3][kC];      // b_t = exp(Lambda_t)
    float beta[3][kC];
    int abort;
    uint32_t tmem;
};
constexpr int kSmem = kCtl + (int)sizeof(Ctl) + 1024;
static_assert(kSmem <= 232448, "fits in one SM's shared memory");
static_assert(kStage % 1024 == 0 && kKt % 1024 == 0 && kGq % 1024 == 0, "operand tiles 1024-byte aligned");

// TMEM columns (512 allocated)
constexpr uint32_t kTx = 0;       // S^T, fp32
constexpr uint32_t kTxh = 128;    // S0^T operand hi (bf16 pairs); lo at +64
constexpr uint32_t kTo1 = 256;    // O1^T accumulator (64 columns)
constexpr uint32_t kTo2 = 320;    // O2^T accumulator
constexpr uint32_t kTg = 384;     // Gram Q K^T (lanes 0..63 = tokens t)

// the 16 tokens cg*16 .. of channel quarter*32 + lane, as bf16 pairs in opk, to o:
// through the warp's staging tile, 8 tokens at a time, each lane storing one
// 16-byte run of 8 channels of one token
__device__ __forceinline__ void store_o(const ScanArgs &a, int h, int cg, int quarter, int lane, int64_t crow,
                                        int nvalid, const uint32_t (&opk)[8], __nv_bfloat16 *stg) {
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.o_out) + (int64_t)h * kD + quarter * 32 + (lane & 3) * 8;
    const int64_t rs = (int64_t)a.H * kD;
    uint16_t *st16 = reinterpret_cast<uint16_t *>(stg);
#pragma unroll
    for (int ps = 0; ps < 2; ++ps) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w = opk[ps * 4 + (i >> 1)];
            st16[i * 32 + lane] = (uint16_t)((i & 1) ? (w >> 16) : (w & 0xFFFFu));
        }
        __syncwarp();
        const int i = lane >> 2;
        const int t = cg * 16 + ps * 8 + i;
        const uint4 val = *reinterpret_cast<const uint4 *>(stg + i * 32 + (lane & 3) * 8);
        if (t < nvalid) *reinterpret_cast<uint4 *>(o + (crow + t) * rs) = val;
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    scan_sd_o_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q, const ScanArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align1024(smem_raw);
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + kCtl);
    volatile int *abortp = &ctl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int unit = blockIdx.x;   // (layer, segment, head)
    const int h = unit % a.H;
    const int seg = (unit / a.H) % a.n_seg;
    const int l = unit / (a.H * a.n_seg);
    int64_t t0 = a.seg_offsets[seg], t1 = a.seg_offsets[seg + 1];
    const bool bad = !(t0 >= 0 && t0 <= t1 && t1 <= a.N);
    if (bad) t0 = t1 = 0;
    const int nc = (int)((t1 - t0 + kC - 1) / kC);
    const int64_t row0 = (int64_t)l * a.N + t0;

    if (threadIdx.x == 0) {
        if (bad) flag_index_error(a.d_err);
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->gram_done, 1);
        mbar_init(&ctl->gk_ready, kCW / 32);
        mbar_init(&ctl->xop_ready, kCW / 32);
        mbar_init(&ctl->x_done, 1);
        mbar_init(&ctl->o_done, 1);
        mbar_init(&ctl->o_free, kCW / 32);
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        mbar_fence_init();
        tma_prefetch(&tm_k);
        tma_prefetch(&tm_v);
        tma_prefetch(&tm_q);
    }
    if (warp == 0) tmem_alloc(&ctl->tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;

    constexpr uint32_t id_g = idesc_bf16_f32(128, 64, false, false);    // Q (K-major) x K (K-major)
    constexpr uint32_t id_o1 = idesc_bf16_f32(128, 64, false, false);   // S0^T (TMEM) x Q (K-major)
    constexpr uint32_t id_x = idesc_bf16_f32(128, 128, true, true);     // V^T (MN-major) x K~ (MN-major)
    constexpr uint32_t id_o2 = idesc_bf16_f32(128, 64, true, false);    // V^T (MN-major) x Gq (K-major)

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            for (int j = 0; j < nc; ++j) {
                const int s = j % kNS;
                if (!wait_or_abort(&ctl->empty[s], ((uint32_t)(j / kNS) & 1u) ^ 1u, abortp)) break;
                uint8_t *st = smem + s * kStage;
                const int row = (int)(row0 + (int64_t)j * kC);
                mbar_expect_tx(&ctl->full[s], (uint32_t)kStage);
                tma_load_3d(st + kOffK, &tm_k, &ctl->full[s], 0, h, row);
                tma_load_3d(st + kOffK + kBox, &tm_k, &ctl->full[s], 64, h, row);
                tma_load_3d(st + kOffV, &tm_v, &ctl->full[s], 0, h, row);
                tma_load_3d(st + kOffV + kBox, &tm_v, &ctl->full[s], 64, h, row);
                tma_load_3d(st + kOffQ, &tm_q, &ctl->full[s], 0, h, row);
                tma_load_3d(st + kOffQ + kBox, &tm_q, &ctl->full[s], 64, h, row);
                issued = j + 1;
            }
            if (*abortp)
                for (int j = issued - kNS < 0 ? 0 : issued - kNS; j < issued; ++j)
                    mbar_wait(&ctl->full[j % kNS], (uint32_t)(j / kNS) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer: per chunk the
        // update first (the chain), then the next chunk's Gram (so its Gq and K~ can be
        // built meanwhile), then the outputs
        if (lane == 0) {
            auto gram = [&](int jj) -> bool {   // G = Q K^T of chunk jj into the Gram columns
                const int s = jj % kNS;
                if (!wait_or_abort(&ctl->full[s], (uint32_t)(jj / kNS) & 1u, abortp)) return false;
                tc_fence_after();
                const uint8_t *stg = smem + s * kStage;
                const uint32_t kb = smem_addr(stg + kOffK), qb = smem_addr(stg + kOffQ);
                const uint64_t dq = smem_desc_sw128(qb, 0, 1024), dk = smem_desc_sw128(kb, 0, 1024);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t o = (uint64_t)((ks >> 2) * (kBox >> 4) + (ks & 3) * 2);
                    mma_f16(tmem + kTg, dq + o, dk + o, id_g, ks > 0 ? 1u : 0u);
                }
                mma_commit(&ctl->gram_done);
                return true;
            };
            bool ok = nc == 0 || gram(0);
            for (int j = 0; j < nc && ok; ++j) {
                const int s = j % kNS;
                const uint32_t par = (uint32_t)j & 1u;
                const uint8_t *stg = smem + s * kStage;
                const uint32_t vb = smem_addr(stg + kOffV), qb = smem_addr(stg + kOffQ);
                // Gq, K~ of this chunk and its S0 operand are in place (S rewritten as b_C S0)
                if (!wait_or_abort(&ctl->gk_ready, par, abortp) || !wait_or_abort(&ctl->xop_ready, par, abortp)) break;
                tc_fence_after();
                // ---- S^T += V^T K~ (lo, then hi)
                const uint32_t kt = smem_addr(smem + kKt);
                const uint64_t dv = smem_desc_sw128(vb, kBox, 1024), dkt = smem_desc_sw128(kt, kBox, 1024),
                               dq = smem_desc_sw128(qb, 0, 1024);
#pragma unroll
                for (int hl = 1; hl >= 0; --hl)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16(tmem + kTx, dv + (uint64_t)(ks * 128), dkt + (uint64_t)(hl * 1024 + ks * 128), id_x,
                                1u);
                mma_commit(&ctl->x_done);
                // ---- the next chunk's Gram (its columns were read for this chunk's Gq)
                if (j + 1 < nc && !gram(j + 1)) break;
                // ---- O1^T = S0^T Q^T, O2^T = V^T Gq^T (lo, then hi), once the previous ones are read
                if (j > 0 && !wait_or_abort(&ctl->o_free, par ^ 1u, abortp)) break;
                tc_fence_after();
#pragma unroll
                for (int hl = 1; hl >= 0; --hl)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (uint32_t)(ks >> 2) * kBox + (uint32_t)(ks & 3) * 32u;
                        mma_f16_ta(tmem + kTo1, tmem + kTxh + (uint32_t)hl * 64u + (uint32_t)ks * 8u,
                                   dq + (uint64_t)(off >> 4), id_o1, (hl == 0 || ks > 0) ? 1u : 0u);
                    }
                const uint64_t dg = smem_desc_sw128(smem_addr(smem + kGq + (int)par * 16384), 0, 1024);
#pragma unroll
                for (int hl = 1; hl >= 0; --hl)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16(tmem + kTo2, dv + (uint64_t)(ks * 128), dg + (uint64_t)(hl * 512 + ks * 2), id_o2,
                                (hl == 0 || ks > 0) ? 1u : 0u);
                mma_commit(&ctl->o_done);
                mma_commit(&ctl->empty[s]);
            }
            if (*abortp) {   // drain: completes once this thread's MMAs are done
                mma_commit(&ctl->drain);
                mbar_wait(&ctl->drain, 0);
            }
        }
    } else {
        // ------------------------------------------------------------ conversion warps
        const int st = threadIdx.x - 64;          // 0..511
        const int sw = warp - 2;                  // 0..15
        const int cg = sw >> 2;                   // column group (16 columns) of this warp
        const int quarter = warp & 3;             // TMEM lanes this warp may touch
        const int m = quarter * 32 + lane;        // TMEM lane: value channel (S^T, O), token (Gram)
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tx = tmem + lane_off + kTx + (uint32_t)(cg * 16);
        const uint32_t txh = tmem + lane_off + kTxh + (uint32_t)(cg * 8);
        __nv_bfloat16 *ostg = reinterpret_cast<__nv_bfloat16 *>(smem + kOst) + sw * 256;
        double lam = 0.0;   // sum of log alpha (thread 0)

        {   // S starts at zero
            uint32_t z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = 0u;
            tmem_st16(tx, z);
            tmem_st16(tx + 64u, z);
            tmem_wait_st();
        }

        // alpha, beta of one chunk (warp 0 of the group, two tokens a lane), loaded a chunk ahead
        float ga[2] = {1.f, 1.f}, gb[2] = {0.f, 0.f};
        auto gate_load = [&](int jj) {
            if (jj >= nc) return;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int t = lane + 32 * q;
                const bool v = (int64_t)jj * kC + t < t1 - t0;
                const int64_t r = (row0 + (int64_t)jj * kC + t) * a.H + h;
                ga[q] = v ? a.alpha[r] : 1.f;
                gb[q] = v ? (a.beta ? a.beta[r] : 1.f) : 0.f;
            }
        };
        if (sw == 0) gate_load(0);
        // gates, Gq and K~ of chunk jj (slot jj % 3, Gq tiles of parity jj & 1); false on a timeout
        auto prep = [&](int jj) -> bool {
            const int gsl = jj % 3;
            const int s = jj % kNS;
            const uint8_t *stg = smem + s * kStage;
            const uint32_t par = (uint32_t)jj & 1u;
            const int nval = (int)min((int64_t)kC, t1 - t0 - (int64_t)jj * kC);
            if (sw == 0) {   // Lambda_t (inclusive log-space prefix), b_t, beta_t
                float lg[2], pb[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const bool v = lane + 32 * q < nval;
                    lg[q] = v ? logf(ga[q]) : 0.f;
                    pb[q] = v ? gb[q] : 0.f;
                }
                gate_load(jj + 1);   // the next chunk's gates, in flight while this one is used
                float inc[2];
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
                inc[1] += __shfl_sync(0xffffffffu, inc[0], 31);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int t = lane + 32 * q;
                    ctl->lt[gsl][t] = inc[q];
                    ctl->bt[gsl][t] = expf(inc[q]);
                    ctl->beta[gsl][t] = pb[q];
                }
                lam += (double)__shfl_sync(0xffffffffu, inc[1], 31);   // lambda: chunk totals in double
            }
            const bool ok = wait_or_abort(&ctl->full[s], (uint32_t)(jj / kNS) & 1u, abortp) &&
                            wait_or_abort(&ctl->gram_done, par, abortp);
            if (!bar_and(2, kCW, ok)) return false;
            tc_fence_after();
            const float LC = ctl->lt[gsl][kC - 1];
            // ---- Gq[t][s] = [s <= t] exp(Lambda_t - Lambda_s) beta_s G[t][s] -> bf16 hi / lo
            // (row t, s contiguous, 128-byte swizzle); lanes 0..63 of the Gram
            if (quarter < 2) {
                const int t = m;
                uint32_t r[16];
                tmem_ld16(tmem + lane_off + kTg + (uint32_t)(cg * 16), r);
                const float ltt = ctl->lt[gsl][t];
                float f[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int sc = cg * 16 + i;
                    f[i] = sc <= t ? __expf(ltt - ctl->lt[gsl][sc]) * ctl->beta[gsl][sc] : 0.f;
                }
                tmem_wait_ld();
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    split_pair(f[2 * q] * __uint_as_float(r[2 * q]), f[2 * q + 1] * __uint_as_float(r[2 * q + 1]), hi[q],
                               lo[q]);
                uint8_t *gt = smem + kGq + (int)par * 16384 + t * 128;
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                    const int c = 2 * cg + hc;
                    const int off = (c ^ (t & 7)) << 4;
                    *reinterpret_cast<uint4 *>(gt + off) =
                        make_uint4(hi[4 * hc], hi[4 * hc + 1], hi[4 * hc + 2], hi[4 * hc + 3]);
                    *reinterpret_cast<uint4 *>(gt + 8192 + off) =
                        make_uint4(lo[4 * hc], lo[4 * hc + 1], lo[4 * hc + 2], lo[4 * hc + 3]);
                }
            }
            // ---- K~_s = exp(LC - Lambda_s) beta_s k_s -> bf16 hi / lo (same swizzled layout as K),
            // once the previous update has read the tiles
            if (!bar_and(2, kCW, jj == 0 || wait_or_abort(&ctl->x_done, par ^ 1u, abortp))) return false;
            {
                const int sidx = st >> 3;           // token
                const int g = st & 7;               // 16-channel group
                const int box = g >> 2;
                const float w = __expf(LC - ctl->lt[gsl][sidx]) * ctl->beta[gsl][sidx];
                uint8_t *kt = smem + kKt;
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                    const int c = (g & 3) * 2 + hc;
                    const int off = box * kBox + sidx * 128 + ((c ^ (sidx & 7)) << 4);
                    const uint4 raw = *reinterpret_cast<const uint4 *>(stg + kOffK + off);
                    const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
                    uint32_t hv[4], lv[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p)
                        split_pair(__uint_as_float(in[p] << 16) * w, __uint_as_float(in[p] & 0xFFFF0000u) * w, hv[p],
                                   lv[p]);
                    *reinterpret_cast<uint4 *>(kt + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                    *reinterpret_cast<uint4 *>(kt + 16384 + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->gk_ready);
            return true;
        };
        // o_t of chunk jj (b_t O1 + O2 -> bf16); O1, O2 complete (o_done awaited)
        auto out_o = [&](int jj, bool release) {
            uint32_t r1[16], r2[16];
            tmem_ld16(tmem + lane_off + kTo1 + (uint32_t)(cg * 16), r1);
            tmem_ld16(tmem + lane_off + kTo2 + (uint32_t)(cg * 16), r2);
            tmem_wait_ld();
            if (release) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->o_free);
            }
            const int psl = jj % 3;
            uint32_t opk[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int t = cg * 16 + 2 * q;
                const __nv_bfloat162 v2 = __floats2bfloat162_rn(
                    fmaf(ctl->bt[psl][t], __uint_as_float(r1[2 * q]), __uint_as_float(r2[2 * q])),
                    fmaf(ctl->bt[psl][t + 1], __uint_as_float(r1[2 * q + 1]), __uint_as_float(r2[2 * q + 1])));
                opk[q] = *reinterpret_cast<const uint32_t *>(&v2);
            }
            store_o(a, h, cg, quarter, lane, row0 + (int64_t)jj * kC, (int)min((int64_t)kC, t1 - t0 - (int64_t)jj * kC),
                    opk, ostg);
        };

        bool alive = nc == 0 || prep(0);
        for (int j = 0; j < nc && alive; ++j) {
            const uint32_t par = (uint32_t)j & 1u;
            // ---- S0 operand (hi / lo) and S <- b_C S0: the previous update and the previous
            // outputs' products (which read the S0 operand) are done
            bool ok = j == 0 || (wait_or_abort(&ctl->x_done, par ^ 1u, abortp) &&
                                 wait_or_abort(&ctl->o_done, par ^ 1u, abortp));
            if (!bar_and(2, kCW, ok)) {
                alive = false;
                break;
            }
            tc_fence_after();
            const float bC = ctl->bt[j % 3][kC - 1];
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                uint32_t r[16], hi[8], lo[8];
                tmem_ld16(tx + (uint32_t)(p * 64), r);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    split_pair(__uint_as_float(r[2 * q]), __uint_as_float(r[2 * q + 1]), hi[q], lo[q]);
                tmem_st8(txh + (uint32_t)(p * 32), hi);
                tmem_st8(txh + 64u + (uint32_t)(p * 32), lo);
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(bC * __uint_as_float(r[i]));
                tmem_st16(tx + (uint32_t)(p * 64), r);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->xop_ready);
            // ---- the previous chunk's outputs, then the next chunk's Gq and K~
            if (j > 0) out_o(j - 1, true);
            if (j + 1 < nc && !prep(j + 1)) {
                alive = false;
                break;
            }
        }
        if (alive && nc > 0) {   // the last chunk's outputs
            if (bar_and(2, kCW, wait_or_abort(&ctl->o_done, (uint32_t)(nc - 1) & 1u, abortp))) {
                tc_fence_after();
                out_o(nc - 1, false);
            } else {
                alive = false;
            }
        }

        // ------------------------------------------------------------ epilogue: the state
        bool ok = alive && (nc == 0 || wait_or_abort(&ctl->x_done, (uint32_t)(nc - 1) & 1u, abortp));
        if (bar_and(2, kCW, ok)) {
            tc_fence_after();
            const int64_t u_out = ((int64_t)l * a.n_seg + seg) * a.H + h;
            uint32_t r[2][16];
            tmem_ld16(tx, r[0]);
            tmem_ld16(tx + 64u, r[1]);
            tmem_wait_ld();
            float *out = a.S_out + u_out * kD * kD;
#pragma unroll
            for (int p = 0; p < 2; ++p)
#pragma unroll
                for (int i = 0; i < 16; ++i) out[(int64_t)(p * 64 + cg * 16 + i) * kD + m] = __uint_as_float(r[p][i]);
            if (st == 0) a.lam_out[u_out] = (float)lam;
        } else {
            *abortp = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abortp && a.d_err) atomicExch(a.d_err, (int)HYPIC_ETIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool scan_sd_o_supported(const ScanArgs &a) {
    return a.fam == HYPIC_SCALAR && a.in_dtype == HYPIC_BF16 && a.dk == kD && a.dv == kD && a.o_out != nullptr &&
           a.q != nullptr && a.N > 0 && (int64_t)a.n_layers * a.N < ((int64_t)1 << 31) &&
           (int64_t)a.n_layers * a.n_seg * a.H < ((int64_t)1 << 31) && tensor_map_encoder() != nullptr;
}

cudaError_t launch_scan_sd_o(const ScanArgs &a, cudaStream_t s) {
    const int64_t units = (int64_t)a.n_layers * a.n_seg * a.H;
    if (units == 0) return cudaSuccess;
    const uint64_t rows = (uint64_t)a.n_layers * (uint64_t)a.N;
    CUtensorMap mk, mv, mq;
    if (!make_tensor_map_3d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k, kD, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v, kD, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, kD, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(scan_sd_o_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    scan_sd_o_kernel<<<(unsigned)units, kThreads, kSmem, s>>>(mk, mv, mq, a);
    return cudaGetLastError();
}

}  // namespace hypic
