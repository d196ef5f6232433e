// scan_diag_o.cu -- diagonal-gated segment scan (a gate per key channel: GLA-style)
// with the per-token outputs o_t on tcgen05 tensor cores, bf16 q / k / v / o,
// d_k = d_v = 128.
//
// Chunks of C = 64 tokens in order.  With Lam_t the inclusive in-chunk prefix sum
// of log alpha per key channel, S0 the state at the chunk's start and L = Lam_63:
//   S_t = diag(e^Lam_t) S0 + sum_{s<=t} beta_s diag(e^(Lam_t - Lam_s)) k_s v_s^T,
//   o_t = S_t^T q_t = (O1 + O2)_t,
//   O1 = Aq (diag(e^ra) S0),   Aq_t = q_t o e^(Lam_t - ra),
//   O2 = Gq V,  Gq[t][s] = [s <= t] sum_i q_ti k_si beta_s e^(Lam_t,i - Lam_s,i),
//   S_C = diag(e^L) S0 + Bk^T V diag-scaled:  with Bk_s = beta_s k_s o e^(rb - Lam_s),
//   X = diag(e^rb) S0 + Bk^T V  and  S_C = diag(e^(L - rb)) X.
// The Gram's decay ratio factors through per-channel references, e^(Lam_t - Lam_s)
// = e^(Lam_t - r) e^(r - Lam_s), so Gq = tril(Aq Bk^T) is one tensor-core product
// when ra = rb = r = Lam_31 (every factor below e^60 while |Lam - r| <= 60 nats).
// A chunk beyond that (a channel that decays by more than e^60 within half a
// chunk) takes ra = 0 and rb = L (Aq and Bk both at most 1) and its Gq exactly on
// CUDA cores.  The state lives in TMEM transposed (lane = value channel j,
// column = key channel i) as X, fp32; each chunk's conversion warps rewrite it as
// diag(e^rb) S0 (S0 = diag(e^(L' - rb')) X' of the chunk before) and split
// diag(e^ra) S0 into the bf16 hi / lo operand of O1.  Per CTA one (layer,
// segment, head):
//   warp 0       TMA: q, k, v of a chunk (two 64-channel boxes each), two stages;
//   warp 1       one thread issues every tcgen05.mma: Gram Aq Bk^T (hi / lo, three
//                products), then X += V^T Bk (Bk split), O1^T = (S0 op)^T Aq^T
//                (both split: three products), O2^T = V^T Gq^T (Gq split);
//   warps 2-17   gates (log-space prefix sums per channel), the Aq / Bk tiles, Gq,
//                the state rewrite and its operand, o_t = O1 + O2 (bf16), the
//                final state and lambda (sum of log alpha per channel).
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
constexpr int kNS = 2;                    // TMA stages
constexpr int kCW = 512;                  // conversion threads (16 warps)
constexpr int kThreads = 64 + kCW;
constexpr float kMaxLog2 = 60.f * 1.4426950408889634f;   // |Lam - r| bound, base 2

// shared memory, from the 1024-aligned base
constexpr int kStage = 6 * kBox;          // q, k, v: two boxes each
constexpr int kOffQ = 0, kOffK = 2 * kBox, kOffV = 4 * kBox;
constexpr int kAq = kNS * kStage;         // Aq hi (two boxes), lo +16 KB
constexpr int kBk = kAq + 32768;          // Bk hi (two boxes), lo +16 KB
constexpr int kGq = kBk + 32768;          // Gq hi (rows t, s along K), lo +8 KB
constexpr int kLam = kGq + 16384;         // Lam, base 2, fp32 [64][128] (row t = Lam_t)
constexpr int kOst = kLam + kC * kD * 4;  // o staging: 8 tokens x 32 channels per warp
constexpr int kCtl = kOst + 16 * 512;

struct Ctl {
    uint64_t full[kNS], empty[kNS];
    uint64_t ops_ready, gram_done, gk_ready, o_done, o_free, drain;
    float beta[kC];
    float ra[kD], rb[kD];       // this chunk's references (base 2)
    float fa[kD], fb[kD];       // rewrite factors e^(ra) g', e^(rb) g' (g' = e^(L' - rb') of the chunk before)
    float g[2][kD];             // e^(L - rb) of chunk j in slot j & 1
    float part[4][kD];          // per-part totals of the prefix
    int steep[2];
    int abort;
    uint32_t tmem;
};
constexpr int kSmem = kCtl + (int)sizeof(Ctl) + 1024;
static_assert(kSmem <= 232448, "fits in one SM's shared memory");
static_assert(kStage % 1024 == 0 && kAq % 1024 == 0 && kBk % 1024 == 0 && kGq % 1024 == 0, "tiles 1024-aligned");

// TMEM columns (512 allocated)
constexpr uint32_t kTx = 0;       // X^T, fp32 (lane = value channel j, column = key channel i)
constexpr uint32_t kTxh = 128;    // O1's A operand, diag(e^ra) S0, bf16 pairs hi; lo at +64
constexpr uint32_t kTo1 = 256;    // O1^T (64 columns)
constexpr uint32_t kTo2 = 320;    // O2^T
constexpr uint32_t kTg = 384;     // Gram Aq Bk^T (lanes 0..63 = tokens t)

__device__ __forceinline__ int swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ void put8(uint8_t *dst, int lo_off, const float (&x)[8]) {
    uint32_t hv[4], lv[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) split_pair(x[2 * p], x[2 * p + 1], hv[p], lv[p]);
    *reinterpret_cast<uint4 *>(dst) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    *reinterpret_cast<uint4 *>(dst + lo_off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
}

__device__ __forceinline__ void load8(const float *p, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ float bf_at(const uint8_t *tile, int row, int ch) {   // one bf16 of a 2-box tile
    const uint16_t b = *reinterpret_cast<const uint16_t *>(tile + (ch >> 6) * kBox + swz(row, (ch & 63) >> 3) +
                                                           ((ch & 7) << 1));
    return __uint_as_float((uint32_t)b << 16);
}

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
    scan_diag_o_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const ScanArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align1024(smem_raw);
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + kCtl);
    float *lam = reinterpret_cast<float *>(smem + kLam);
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
        mbar_init(&ctl->ops_ready, kCW / 32);
        mbar_init(&ctl->gram_done, 1);
        mbar_init(&ctl->gk_ready, kCW / 32);
        mbar_init(&ctl->o_done, 1);
        mbar_init(&ctl->o_free, kCW / 32);
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        mbar_fence_init();
        tma_prefetch(&tm_q);
        tma_prefetch(&tm_k);
        tma_prefetch(&tm_v);
    }
    if (warp == 0) tmem_alloc(&ctl->tmem, 512);
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
                mbar_expect_tx(&ctl->full[s], (uint32_t)kStage);
                tma_load_3d(st + kOffQ, &tm_q, &ctl->full[s], 0, h, row);
                tma_load_3d(st + kOffQ + kBox, &tm_q, &ctl->full[s], 64, h, row);
                tma_load_3d(st + kOffK, &tm_k, &ctl->full[s], 0, h, row);
                tma_load_3d(st + kOffK + kBox, &tm_k, &ctl->full[s], 64, h, row);
                tma_load_3d(st + kOffV, &tm_v, &ctl->full[s], 0, h, row);
                tma_load_3d(st + kOffV + kBox, &tm_v, &ctl->full[s], 64, h, row);
                issued = j + 1;
            }
            if (*abortp)
                for (int j = issued - kNS < 0 ? 0 : issued - kNS; j < issued; ++j)
                    mbar_wait(&ctl->full[j % kNS], (uint32_t)(j / kNS) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_g = idesc_bf16_f32(128, 64, false, false);    // Aq (K-major) x Bk (K-major)
            constexpr uint32_t id_o1 = idesc_bf16_f32(128, 64, false, false);   // S0 op^T (TMEM) x Aq (K-major)
            constexpr uint32_t id_x = idesc_bf16_f32(128, 128, true, true);     // V^T (MN-major) x Bk (MN-major)
            constexpr uint32_t id_o2 = idesc_bf16_f32(128, 64, true, false);    // V^T (MN-major) x Gq (K-major)
            const uint32_t aq = smem_addr(smem + kAq), bk = smem_addr(smem + kBk), gq = smem_addr(smem + kGq);
            const int order[3][2] = {{1, 0}, {0, 1}, {0, 0}};   // lo products first
            // descriptors built once; an operand offset of o bytes adds o >> 4
            const uint64_t daq = smem_desc_sw128(aq, 0, 1024), dbk = smem_desc_sw128(bk, 0, 1024),
                           dbkx = smem_desc_sw128(bk, kBox, 1024), dgq = smem_desc_sw128(gq, 0, 1024);
            for (int j = 0; j < nc; ++j) {
                const int s = j % kNS;
                const uint32_t par = (uint32_t)j & 1u;
                if (!wait_or_abort(&ctl->ops_ready, par, abortp)) break;
                tc_fence_after();
                if (!ctl->steep[par]) {   // Gram Aq Bk^T (M = 128: rows 64..127 unused)
#pragma unroll
                    for (int p = 0; p < 3; ++p)
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint32_t off = (uint32_t)(ks >> 2) * kBox + (uint32_t)(ks & 3) * 32u;
                            mma_f16(tmem + kTg, daq + (uint64_t)((order[p][0] * 16384 + (int)off) >> 4),
                                    dbk + (uint64_t)((order[p][1] * 16384 + (int)off) >> 4), id_g,
                                    (p > 0 || ks > 0) ? 1u : 0u);
                        }
                }
                mma_commit(&ctl->gram_done);
                // Gq, the rewritten state and its operand are in place; the previous outputs read
                if (!wait_or_abort(&ctl->gk_ready, par, abortp) || !wait_or_abort(&ctl->full[s], (uint32_t)(j / kNS) & 1u, abortp) ||
                    (j > 0 && !wait_or_abort(&ctl->o_free, par ^ 1u, abortp)))
                    break;
                tc_fence_after();
                const uint32_t vb = smem_addr(smem + s * kStage + kOffV);
                const uint64_t dv = smem_desc_sw128(vb, kBox, 1024);
                // ---- X^T += V^T Bk (lo, then hi)
#pragma unroll
                for (int hl = 1; hl >= 0; --hl)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16(tmem + kTx, dv + (uint64_t)(ks * 128), dbkx + (uint64_t)(hl * 1024 + ks * 128), id_x, 1u);
                // ---- O1^T = (S0 op)^T Aq^T, both split
#pragma unroll
                for (int p = 0; p < 3; ++p)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (uint32_t)(ks >> 2) * kBox + (uint32_t)(ks & 3) * 32u;
                        mma_f16_ta(tmem + kTo1, tmem + kTxh + (uint32_t)order[p][0] * 64u + (uint32_t)ks * 8u,
                                   daq + (uint64_t)((order[p][1] * 16384 + (int)off) >> 4), id_o1,
                                   (p > 0 || ks > 0) ? 1u : 0u);
                    }
                // ---- O2^T = V^T Gq^T (lo, then hi)
#pragma unroll
                for (int hl = 1; hl >= 0; --hl)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16(tmem + kTo2, dv + (uint64_t)(ks * 128), dgq + (uint64_t)(hl * 512 + ks * 2), id_o2,
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
        const int m = quarter * 32 + lane;        // TMEM lane: value channel (X^T, O), token (Gram)
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tx = tmem + lane_off + kTx + (uint32_t)(cg * 16);
        const uint32_t txh = tmem + lane_off + kTxh + (uint32_t)(cg * 8);
        __nv_bfloat16 *ostg = reinterpret_cast<__nv_bfloat16 *>(smem + kOst) + sw * 256;
        const int ch = st & (kD - 1), part = st >> 7;   // gates: channel, 16-token part
        double lam_acc = 0.0;                            // lambda of channel ch (part 0)

        {   // X starts at zero
            uint32_t z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = 0u;
            tmem_st16(tx, z);
            tmem_st16(tx + 64u, z);
            tmem_wait_st();
        }

        // alpha of chunk jj for this thread's channel and part (16 tokens), beta (part 0,
        // lanes of warp 0: two tokens each)
        float ga[16], gbeta[2];
        auto gate_load = [&](int jj) {
            if (jj >= nc) return;
            const int64_t base = row0 + (int64_t)jj * kC;
            const int nv = (int)min((int64_t)kC, t1 - t0 - (int64_t)jj * kC);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t = part * 16 + i;
                ga[i] = t < nv ? a.alpha[((base + t) * a.H + h) * kD + ch] : 1.f;
            }
            if (sw == 0) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int t = lane + 32 * q;
                    gbeta[q] = t < nv ? (a.beta ? a.beta[(base + t) * a.H + h] : 1.f) : 0.f;
                }
            }
        };
        // Lam, references and factors of chunk jj from the loaded gates (true: finite)
        auto gates = [&](int jj) -> bool {
            const uint32_t par = (uint32_t)jj & 1u;
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                acc += log2f(ga[i]);
                lam[(part * 16 + i) * kD + ch] = acc;
            }
            ctl->part[part][ch] = acc;
            if (sw == 0) {
                ctl->beta[lane] = gbeta[0];
                ctl->beta[lane + 32] = gbeta[1];
            }
            bar_sync(2, kCW);
            float base = 0.f;
            for (int q = 0; q < part; ++q) base += ctl->part[q][ch];
            float mx = 0.f;
            if (part > 0) {
#pragma unroll
                for (int i = 0; i < 16; ++i) lam[(part * 16 + i) * kD + ch] += base;
            }
            bar_sync(2, kCW);
            const float r = lam[31 * kD + ch];
#pragma unroll
            for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(lam[(part * 16 + i) * kD + ch] - r));
            const bool fine = bar_and(2, kCW, mx <= kMaxLog2);   // false also for a NaN gate
            if (part == 0) {
                const float L = lam[63 * kD + ch];
                const float ra = fine ? r : 0.f, rb = fine ? r : L;
                const float gp = jj > 0 ? ctl->g[par ^ 1u][ch] : 1.f;
                ctl->ra[ch] = ra;
                ctl->rb[ch] = rb;
                ctl->fa[ch] = exp2f(ra) * gp;
                ctl->fb[ch] = exp2f(rb) * gp;
                ctl->g[par][ch] = exp2f(L - rb);
                lam_acc += (double)L * 0.6931471805599453;
                if (ch == 0) ctl->steep[par] = fine ? 0 : 1;
            }
            bar_sync(2, kCW);
            return true;
        };
        // o_t of chunk jj (O1 + O2 -> bf16); O1, O2 complete (o_done awaited)
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
            uint32_t opk[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const __nv_bfloat162 v2 =
                    __floats2bfloat162_rn(__uint_as_float(r1[2 * q]) + __uint_as_float(r2[2 * q]),
                                          __uint_as_float(r1[2 * q + 1]) + __uint_as_float(r2[2 * q + 1]));
                opk[q] = *reinterpret_cast<const uint32_t *>(&v2);
            }
            store_o(a, h, cg, quarter, lane, row0 + (int64_t)jj * kC, (int)min((int64_t)kC, t1 - t0 - (int64_t)jj * kC),
                    opk, ostg);
        };

        bool alive = true;
        gate_load(0);
        if (nc > 0) gates(0);
        for (int j = 0; j < nc && alive; ++j) {
            const int s = j % kNS;
            const uint32_t par = (uint32_t)j & 1u;
            const uint8_t *stg = smem + s * kStage;
            gate_load(j + 1);   // in flight while this chunk is worked on
            // ---- the previous chunk's products are done: its outputs, then its tiles are free
            bool ok = j == 0 || wait_or_abort(&ctl->o_done, par ^ 1u, abortp);
            if (!bar_and(2, kCW, ok)) {
                alive = false;
                break;
            }
            tc_fence_after();
            if (j > 0) out_o(j - 1, true);
            // ---- Aq = q o e^(Lam - ra), Bk = beta k o e^(rb - Lam) -> bf16 hi / lo
            if (!bar_and(2, kCW, wait_or_abort(&ctl->full[s], (uint32_t)(j / kNS) & 1u, abortp))) {
                alive = false;
                break;
            }
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int f = st + kCW * it;   // 0 .. 1023
                const int t = f >> 4, cc = f & 15, b = cc >> 3, c = cc & 7, c8 = cc * 8;
                const int off = b * kBox + swz(t, c);
                const uint4 qr = *reinterpret_cast<const uint4 *>(stg + kOffQ + off);
                const uint4 kr = *reinterpret_cast<const uint4 *>(stg + kOffK + off);
                const uint32_t qw[4] = {qr.x, qr.y, qr.z, qr.w}, kw[4] = {kr.x, kr.y, kr.z, kr.w};
                float lt[8], ra[8], rb[8];
                load8(lam + t * kD + c8, lt);
                load8(ctl->ra + c8, ra);
                load8(ctl->rb + c8, rb);
                const float bt = ctl->beta[t];
                float xa[8], xb[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float qv = __uint_as_float((e & 1) ? (qw[e >> 1] & 0xFFFF0000u) : (qw[e >> 1] << 16));
                    const float kv = __uint_as_float((e & 1) ? (kw[e >> 1] & 0xFFFF0000u) : (kw[e >> 1] << 16));
                    xa[e] = qv * exp2f(lt[e] - ra[e]);
                    xb[e] = bt * kv * exp2f(rb[e] - lt[e]);
                }
                put8(smem + kAq + off, 16384, xa);
                put8(smem + kBk + off, 16384, xb);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->ops_ready);
            // ---- Gq[t][s] = [s <= t] (Aq Bk^T)[t][s], or exactly on CUDA cores (steep chunk)
            ok = wait_or_abort(&ctl->gram_done, par, abortp);
            if (!bar_and(2, kCW, ok)) {
                alive = false;
                break;
            }
            tc_fence_after();
            if (!ctl->steep[par]) {
                if (quarter < 2) {
                    const int t = m;
                    uint32_t r[16];
                    tmem_ld16(tmem + lane_off + kTg + (uint32_t)(cg * 16), r);
                    tmem_wait_ld();
                    float x[2][8];
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[i >> 3][i & 7] = cg * 16 + i <= t ? __uint_as_float(r[i]) : 0.f;
                    put8(smem + kGq + swz(t, 2 * cg), 8192, x[0]);
                    put8(smem + kGq + swz(t, 2 * cg + 1), 8192, x[1]);
                }
            } else {
                // 64 rows x 8 column chunks: Gq[t][s] = sum_i q_ti k_si beta_s 2^(Lam_t,i - Lam_s,i), s <= t
                for (int f = st; f < kC * 8; f += kCW) {
                    const int t = f >> 3, c = f & 7;
                    float x[8];
#pragma unroll 1
                    for (int e = 0; e < 8; ++e) {
                        const int sc = c * 8 + e;
                        float acc = 0.f;
                        if (sc <= t) {
#pragma unroll 4
                            for (int i = 0; i < kD; ++i)
                                acc += bf_at(stg + kOffQ, t, i) * bf_at(stg + kOffK, sc, i) *
                                       exp2f(lam[t * kD + i] - lam[sc * kD + i]);
                            acc *= ctl->beta[sc];
                        }
                        x[e] = acc;
                    }
                    put8(smem + kGq + swz(t, c), 8192, x);
                }
            }
            // ---- X <- e^rb g' o X (= e^rb S0) and O1's operand e^ra g' o X (= e^ra S0), hi / lo
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                uint32_t r[16], hi[8], lo[8];
                tmem_ld16(tx + (uint32_t)(p * 64), r);
                tmem_wait_ld();
                float fa[16], fb[16];
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 va = *reinterpret_cast<const float4 *>(ctl->fa + p * 64 + cg * 16 + i);
                    const float4 vb = *reinterpret_cast<const float4 *>(ctl->fb + p * 64 + cg * 16 + i);
                    fa[i] = va.x; fa[i + 1] = va.y; fa[i + 2] = va.z; fa[i + 3] = va.w;
                    fb[i] = vb.x; fb[i + 1] = vb.y; fb[i + 2] = vb.z; fb[i + 3] = vb.w;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    split_pair(fa[2 * q] * __uint_as_float(r[2 * q]), fa[2 * q + 1] * __uint_as_float(r[2 * q + 1]),
                               hi[q], lo[q]);
                tmem_st8(txh + (uint32_t)(p * 32), hi);
                tmem_st8(txh + 64u + (uint32_t)(p * 32), lo);
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(fb[i] * __uint_as_float(r[i]));
                tmem_st16(tx + (uint32_t)(p * 64), r);
            }
            tmem_wait_st();
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->gk_ready);
            // ---- the next chunk's gates (Lam is free: this chunk's tiles are built)
            if (j + 1 < nc) {
                bar_sync(2, kCW);   // every warp is past its reads of Lam, rb and the factors
                gates(j + 1);
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

        // ------------------------------------------------------------ epilogue: S = e^(L - rb) o X, lambda
        if (bar_and(2, kCW, alive)) {
            const int64_t u_out = ((int64_t)l * a.n_seg + seg) * a.H + h;
            const float *g = ctl->g[(uint32_t)(nc - 1) & 1u];
            uint32_t r[2][16];
            tmem_ld16(tx, r[0]);
            tmem_ld16(tx + 64u, r[1]);
            tmem_wait_ld();
            float *out = a.S_out + u_out * kD * kD;
#pragma unroll
            for (int p = 0; p < 2; ++p)
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int kc = p * 64 + cg * 16 + i;
                    out[(int64_t)kc * kD + m] = (nc > 0 ? g[kc] : 1.f) * __uint_as_float(r[p][i]);
                }
            if (part == 0) a.lam_out[u_out * kD + ch] = (float)lam_acc;
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

bool scan_diag_o_supported(const ScanArgs &a) {
    return a.fam == HYPIC_DIAG && a.in_dtype == HYPIC_BF16 && a.dk == kD && a.dv == kD && a.o_out != nullptr &&
           a.q != nullptr && a.N > 0 && (int64_t)a.n_layers * a.N < ((int64_t)1 << 31) &&
           (int64_t)a.n_layers * a.n_seg * a.H < ((int64_t)1 << 31) && tensor_map_encoder() != nullptr;
}

cudaError_t launch_scan_diag_o(const ScanArgs &a, cudaStream_t s) {
    const int64_t units = (int64_t)a.n_layers * a.n_seg * a.H;
    if (units == 0) return cudaSuccess;
    const uint64_t rows = (uint64_t)a.n_layers * (uint64_t)a.N;
    CUtensorMap mq, mk, mv;
    if (!make_tensor_map_3d(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, kD, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k, kD, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v, kD, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(scan_diag_o_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    scan_diag_o_kernel<<<(unsigned)units, kThreads, kSmem, s>>>(mq, mk, mv, a);
    return cudaGetLastError();
}

}  // namespace hypic
