// scan_dense_ws.cu -- gated delta rule segment scan in two passes over a
// caller-owned workspace: a chunk-parallel preparation pass and the state pass,
// optionally with the per-token outputs o_t = S_t^T q_t.
//
// Chunked WY/UT form of S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
// (C = 64 tokens per chunk; b_t = in-chunk cumulative decay, b_C its total):
//   L_ts = beta_t (b_t / b_s) k_t.k_s  (s < t),   A = (I + L)^-1
//   W = A diag(beta b) K,   U = A diag(beta) V
//   for X = [M | S] (transition and state side by side, d x 2d):
//   Delta = [0 | U] - W X_0,   X <- b_C X_0 + K^T diag(b_C / b) Delta.
// (Within a chunk delta_t = beta_t (v_t - alpha_t S_{t-1}^T k_t) satisfies
// (I + L) Delta = diag(beta) V - diag(beta b) K S_0.)
// Outputs: S_t = b_t S_0 + sum_{s<=t} (b_t / b_s) k_s delta_s^T, so
//   o_t = b_t S_0^T q_t + sum_{s<=t} (b_t / b_s)(q_t.k_s) delta_s
//       = b_t (O1)_t + (O2)_t,  O1 = S_0^T Q^T,  O2 = Delta^T Gq^T,
//   Gq[t][s] = [s <= t] (b_t / b_s) q_t.k_s.
//
// Pass 1 (dense_prep_kernel) depends only on a chunk's own keys, queries and
// gates, so every chunk of every (layer, segment, head) runs in parallel: gates,
// the Gram matrix [K; Q] K^T on tcgen05, L, Gq, and the blocked inverse A,
// written to one workspace record per chunk.  Pass 2 (dense_state_kernel) walks
// the chunks of a chain in order with X^T in TMEM (two CTAs per chain:
// transition half, state half):
//   W^T = K^T (A diag(beta b))^T, U^T = V^T (A diag(beta))^T  (A split bf16 hi + lo)
//   Delta^T = U^T - X0^T W^T    (X0 and W each split hi + lo: three products)
//   X^T    += Delta~^T K        (Delta~ = Delta diag(b_C / b), split hi + lo)
//   O1^T = X0^T Q^T (X0 hi + lo),  O2^T = Delta^T Gq^T (three products)
// W and U are built by their own warps ahead of the state warps; one more warp
// issues the state pass's products, starting on each half of X0 as soon as it
// is converted, and a second issuing warp takes the second k half of Delta (or,
// with o_t, the output products O1 and O2).
#include "dense_common.cuh"
#include "internal.cuh"
#include "sm100.cuh"

namespace hypic {
namespace {

using namespace sm100;
using dense::exponent_of;
using dense::kC;
using dense::kLd;
using dense::split_pair;
using dense::wait_or_abort;

constexpr int kD = 128;
constexpr int kBox = kC * 128;   // 64 channels x 64 tokens, bf16: 8 KB

// ---------------------------------------------------------------- workspace record
// One record per (layer, head, chunk slot), floats.  Without o_t:
//   [0, 8192)        -W^T as bf16 hi / lo operand tiles (row k of 128, tokens t
//                    contiguous, 128-byte swizzle), 16 KB each
//   [8192, 12288)    A diag(beta) as bf16 hi / lo operand tiles (row t, s
//                    contiguous, 128-byte swizzle), 8 KB each
//   G = 12288        gates (below)
// With o_t:
//   [0, 4096)        A diag(beta b) as bf16 hi / lo operand tiles, 8 KB each
//   [4096, 8192)     A diag(beta), the same way
//   G = 8192         gates, then
//   G + 196 + t      b_t
//   [G + 260, +4096) Gq as bf16 hi / lo operand tiles (row t, s contiguous,
//                    128-byte swizzle), 8 KB each
// Gates without o_t: G + t  b_C / b_t;  G + 64, G + 65  log b_C, b_C.
// Gates with o_t: G + t  b_C / b_t;  G + 64 + t  beta_t b_t;  G + 128 + t  beta_t;
//        G + 192, G + 193  log b_C, b_C.
// The state pass stages the head of a record (all but Gq) with the chunk's keys;
// Gq has a buffer of its own.  Chunk j of segment s (tokens from t0) uses slot
// s + floor(t0 / 64) + j, so the slots of different segments never collide and a
// (layer, head) needs at most n_seg + floor(N / 64) of them.
template <bool O>
struct Rec {
    static constexpr int Wt = 0;                            // without o_t
    static constexpr int Abb = 0;                           // with o_t
    static constexpr int Ab = O ? 4096 : 8192;
    static constexpr int G = O ? 8192 : 12288;
    static constexpr int Gw = G;
    static constexpr int Gbb = G + 64, Gbeta = G + 128, B = G + 196;   // with o_t
    static constexpr int LC = O ? G + 192 : G + 64, BC = LC + 1;
    static constexpr int Head = O ? G + 260 : G + 68;      // floats staged with the chunk (multiples of 4)
    static constexpr int Gq = G + 260;                      // with o_t
    static constexpr int Floats = O ? Gq + 4096 : Head;
    static constexpr int Bytes = Floats * 4;                // 49424 / 50192
    static constexpr int HeadBytes = Head * 4;              // 49424 / 33808
    static constexpr int GateFloats = Head - G;             // without o_t: b_C / b, log b_C, b_C (68)
};

__host__ __device__ inline int64_t n_slots(int64_t N, int n_seg) { return (int64_t)n_seg + N / kC; }

// ================================================================ pass 1: preparation

constexpr int kPThreads = 128;
// shared memory (from the 1024-aligned base): the Gram's A operand rows per
// 64-channel box, keys 0..63 then queries 64..127 (without o_t the keys again,
// so that every TMEM lane quarter holds K K^T rows and all four warps share the
// L work).  Once the Gram is done the fp32 L and A tiles overlay that region,
// then temporaries and control: 39.5 KB, five CTAs per SM.
constexpr int kPK = 0;                        // K0 | Q0 (or K0) | K1 | Q1 (or K1)
constexpr int kPAw = kC * kLd * 4;            // L at [0, kPAw), A after it
constexpr int kPTw = kPAw + kC * kLd * 4;
constexpr int kPCtl = kPTw + 3 * 256 * 4;
// without o_t: the keys again for W^T (over L once the inverse is done) and the
// A diag(beta b) operand tiles (over A once every thread has read its part)
constexpr int kPW = 0;
constexpr int kPAb = kPAw;
constexpr int kPWst = 0;                      // then -W^T hi / lo (32 KB) staged for the bulk copy
static_assert(kPTw >= 4 * kBox, "the Gram operands end before the temporaries");
static_assert(kPW + 2 * kBox <= kPAw, "the keys of W^T fit in L's region");
static_assert(kPAb % 1024 == 0 && kPAb + 2 * kBox <= kPTw, "the A diag(beta b) tiles fit in A's region");
static_assert(kPWst + 32768 <= kPTw, "the staged -W^T tiles end before the temporaries");

struct PrepCtl {
    uint64_t full, mma;
    uint32_t tmem;
    float gl[kC], gbeta[kC], gbb[kC];
};
constexpr int kPSmem = kPCtl + (int)sizeof(PrepCtl) + 1024;

template <bool O>
__global__ void __launch_bounds__(kPThreads) dense_prep_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                               const __grid_constant__ CUtensorMap tm_q,
                                                               const ScanArgs a, int64_t slots) {
    using R = Rec<O>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align1024(smem_raw);
    PrepCtl *ctl = reinterpret_cast<PrepCtl *>(smem + kPCtl);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = (int)(blockIdx.x % (unsigned)a.H);
    const int64_t slot = blockIdx.x / (unsigned)a.H;
    const int l = blockIdx.y;

    // slot -> (segment, chunk): the last segment s with s + floor(t0_s / 64) <= slot
    int lo = 0, hi = a.n_seg - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)mid + a.seg_offsets[mid] / kC <= slot) lo = mid;
        else hi = mid - 1;
    }
    const int seg = lo;
    const int64_t t0 = a.seg_offsets[seg], t1 = a.seg_offsets[seg + 1];
    if (!(t0 >= 0 && t0 <= t1 && t1 <= a.N)) return;   // the state pass flags it
    const int64_t j = slot - (seg + t0 / kC);
    if (j < 0 || j * kC >= t1 - t0) return;            // a slot no chunk uses
    const int64_t c0 = t0 + j * kC;                     // first token of the chunk
    float *rec = a.ws + ((int64_t)l * a.H + h) * slots * R::Floats + slot * R::Floats;

    if (tid == 0) {
        mbar_init(&ctl->full, 1);
        mbar_init(&ctl->mma, 1);
        mbar_fence_init();
        mbar_expect_tx(&ctl->full, 4 * kBox);
        const int row = (int)((int64_t)l * a.N + c0);
        tma_load_3d(smem + kPK, &tm_k, &ctl->full, 0, h, row);
        tma_load_3d(smem + kPK + 2 * kBox, &tm_k, &ctl->full, 64, h, row);
        tma_load_3d(smem + kPK + kBox, O ? &tm_q : &tm_k, &ctl->full, 0, h, row);
        tma_load_3d(smem + kPK + 3 * kBox, O ? &tm_q : &tm_k, &ctl->full, 64, h, row);
    }
    if (warp == 0) tmem_alloc(&ctl->tmem, 64);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    bool ok = true;

    // ---- Gram [K; Q] K^T as soon as the keys are in (warp 0): lanes 0..63 K K^T,
    // lanes 64..127 Q K^T (K K^T again without o_t); the gates meanwhile (warp 1)
    if (warp == 0 && lane == 0) {
        ok = mbar_wait(&ctl->full, 0);
        if (ok) {
            tc_fence_after();
            constexpr uint32_t id_gram = idesc_bf16_f32(128, 64, false, false);
            const uint32_t kb = smem_addr(smem + kPK);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (uint32_t)(ks >> 2) * (2u * kBox) + (uint32_t)(ks & 3) * 32u;
                const uint64_t d = smem_desc_sw128(kb + off, 0, 1024);
                mma_f16(tmem, d, d, id_gram, ks > 0);
            }
        }
        mma_commit(&ctl->mma);
    }
    // ---- gates (warp 1): Lambda, b_C / b, beta b, beta, log b_C, b_C (, b)
    if (warp == 1) {
        float lg[2], pb[2], inc[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int64_t t = c0 + lane + 32 * q;
            const bool v = t < t1;
            const int64_t row = ((int64_t)l * a.N + t) * a.H + h;
            lg[q] = v ? logf(a.alpha[row]) : 0.f;
            pb[q] = v ? (a.beta ? a.beta[row] : 1.f) : 0.f;
        }
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
        const float total = __shfl_sync(0xffffffffu, inc[1], 31);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int t = lane + 32 * q;
            const float bt = expf(inc[q]);
            ctl->gl[t] = inc[q];
            ctl->gbeta[t] = pb[q];
            ctl->gbb[t] = pb[q] * bt;
            rec[R::Gw + t] = expf(total - inc[q]);
            if (O) {
                rec[R::Gbb + t] = pb[q] * bt;
                rec[R::Gbeta + t] = pb[q];
                rec[R::B + t] = bt;
            }
        }
        if (lane == 0) {
            rec[R::LC] = total;
            rec[R::BC] = expf(total);
            if (!O) rec[R::BC + 1] = rec[R::BC + 2] = 0.f;
        }
    }
    ok = __syncthreads_and(ok && mbar_wait(&ctl->mma, 0));
    tc_fence_after();
    float *Lw = reinterpret_cast<float *>(smem + kPK);
    float *Aw = reinterpret_cast<float *>(smem + kPAw);
    float *Tw = reinterpret_cast<float *>(smem + kPTw);
    if (ok) {
        const int t = (warp & 1) * 32 + lane;   // token row 0..63 of this thread
        const float lt = ctl->gl[t];
        if (!O) {
            // ---- L[t][s] = beta_t exp(Lambda_t - Lambda_s) G[t][s] for s < t; warps 0, 1
            // take columns 0..31, warps 2, 3 columns 32..63 (from the second copy)
            const float bt = ctl->gbeta[t];
            const int cbase = (warp >> 1) * 32;
            uint32_t r[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)cbase, r);
            float gs[32];   // all loads before the first store (the L tile could alias them)
#pragma unroll
            for (int i = 0; i < 32; ++i) gs[i] = ctl->gl[cbase + i];
            tmem_wait_ld();
            // 16-byte stores: rows are kLd floats apart, so 4-byte stores of one column
            // by the warp's 32 rows would hit 8 banks four times over
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                float4 v;
                float *vp = &v.x;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int sc = cbase + i + e;
                    vp[e] = sc < t ? bt * __expf(lt - gs[i + e]) * __uint_as_float(r[i + e]) : 0.f;
                }
                *reinterpret_cast<float4 *>(Lw + t * kLd + cbase + i) = v;
            }
        } else if (warp < 2) {
            // ---- L[t][s] = beta_t exp(Lambda_t - Lambda_s) G[t][s] for s < t
            const float bt = ctl->gbeta[t];
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(cb * 32), r);
                float gs[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) gs[i] = ctl->gl[cb * 32 + i];
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    float4 v;
                    float *vp = &v.x;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int sc = cb * 32 + i + e;
                        vp[e] = sc < t ? bt * __expf(lt - gs[i + e]) * __uint_as_float(r[i + e]) : 0.f;
                    }
                    *reinterpret_cast<float4 *>(Lw + t * kLd + cb * 32 + i) = v;
                }
            }
        } else if (O) {
            // ---- Gq -> bf16 hi / lo tiles: the state pass multiplies it with Delta~_s =
            // fD (b_C / b_s) Delta_s, so Gq[t][s] = [s <= t] (b_t / b_C) (q_t.k_s) (the
            // factor of s cancels); a chunk that decays below e^-40 keeps Delta_s itself
            // there (Delta~ may underflow) and takes Gq[t][s] = [s <= t] (b_t / b_s) (q_t.k_s)
            uint8_t *gq = reinterpret_cast<uint8_t *>(rec + R::Gq);
            const float lc = ctl->gl[kC - 1];    // log b_C
            const bool steep = lc < -40.f;
            const float rt = __expf(lt - lc);   // b_t / b_C
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(cb * 32), r);
                float gs[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) gs[i] = ctl->gl[cb * 32 + i];
                tmem_wait_ld();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c = cb * 4 + cc;
                    uint32_t hv[4], lv[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        float x[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int sc = c * 8 + 2 * p + e;
                            const float f = steep ? __expf(lt - gs[cc * 8 + 2 * p + e]) : rt;
                            x[e] = sc <= t ? f * __uint_as_float(r[cc * 8 + 2 * p + e]) : 0.f;
                        }
                        split_pair(x[0], x[1], hv[p], lv[p]);
                    }
                    const int off = t * 128 + ((c ^ (t & 7)) << 4);
                    *reinterpret_cast<uint4 *>(gq + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                    *reinterpret_cast<uint4 *>(gq + 8192 + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
                }
            }
        }
        if (!O) fence_async_smem();   // L's region takes the keys again (async proxy) after the inverse
        __syncthreads();
        dense::tri_inverse<kPThreads, 1, false, true>(Lw, Aw, Tw, tid);
        if (!O && tid == 0) {
            // the keys again for W^T, into L's dead region, while the tiles are built
            mbar_expect_tx(&ctl->full, 2 * kBox);
            const int row = (int)((int64_t)l * a.N + c0);
            tma_load_3d(smem + kPW, &tm_k, &ctl->full, 0, h, row);
            tma_load_3d(smem + kPW + kBox, &tm_k, &ctl->full, 64, h, row);
        }
        if (O) {
            // ---- A diag(beta b) and A diag(beta) -> bf16 hi / lo tiles in the record (row t,
            // 8-column group c at 16-byte position c ^ (t & 7); zero above the diagonal blocks)
            uint8_t *tiles = reinterpret_cast<uint8_t *>(rec + R::Abb);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int f = tid + kPThreads * i;   // 0 .. 511
                const int tt = f >> 3, c = f & 7;
                float x[8];
                if ((c >> 1) > (tt >> 4)) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = 0.f;
                } else {
                    const float4 x0 = *reinterpret_cast<const float4 *>(Aw + tt * kLd + c * 8);
                    const float4 x1 = *reinterpret_cast<const float4 *>(Aw + tt * kLd + c * 8 + 4);
                    x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
                    x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
                }
                const int off = tt * 128 + ((c ^ (tt & 7)) << 4);
                uint32_t hv[4], lv[4];
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    split_pair(x[2 * p] * ctl->gbb[c * 8 + 2 * p], x[2 * p + 1] * ctl->gbb[c * 8 + 2 * p + 1], hv[p],
                               lv[p]);
                *reinterpret_cast<uint4 *>(tiles + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                *reinterpret_cast<uint4 *>(tiles + 8192 + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    split_pair(x[2 * p] * ctl->gbeta[c * 8 + 2 * p], x[2 * p + 1] * ctl->gbeta[c * 8 + 2 * p + 1],
                               hv[p], lv[p]);
                *reinterpret_cast<uint4 *>(tiles + 16384 + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                *reinterpret_cast<uint4 *>(tiles + 24576 + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
            }
        } else {
            // ---- A diag(beta) -> bf16 hi / lo tiles in the record, A diag(beta b) -> hi / lo
            // tiles in shared memory over A itself (the operand of W^T): every thread reads its
            // A values first (row t, 8-column group c at 16-byte position c ^ (t & 7); zero
            // above the diagonal blocks)
            uint8_t *tiles = reinterpret_cast<uint8_t *>(rec + R::Ab);
            uint32_t wh[4][4], wl[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int f = tid + kPThreads * i;   // 0 .. 511
                const int tt = f >> 3, c = f & 7;
                float x[8];
                if ((c >> 1) > (tt >> 4)) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = 0.f;
                } else {
                    const float4 x0 = *reinterpret_cast<const float4 *>(Aw + tt * kLd + c * 8);
                    const float4 x1 = *reinterpret_cast<const float4 *>(Aw + tt * kLd + c * 8 + 4);
                    x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
                    x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
                }
                const int off = tt * 128 + ((c ^ (tt & 7)) << 4);
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    split_pair(x[2 * p] * ctl->gbb[c * 8 + 2 * p], x[2 * p + 1] * ctl->gbb[c * 8 + 2 * p + 1],
                               wh[i][p], wl[i][p]);
                uint32_t hv[4], lv[4];
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    split_pair(x[2 * p] * ctl->gbeta[c * 8 + 2 * p], x[2 * p + 1] * ctl->gbeta[c * 8 + 2 * p + 1],
                               hv[p], lv[p]);
                *reinterpret_cast<uint4 *>(tiles + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                *reinterpret_cast<uint4 *>(tiles + 8192 + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
            }
            __syncthreads();   // A (fp32) is read for the last time
            uint8_t *wop = smem + kPAb;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int f = tid + kPThreads * i;
                const int tt = f >> 3, c = f & 7;
                const int off = tt * 128 + ((c ^ (tt & 7)) << 4);
                *reinterpret_cast<uint4 *>(wop + off) = make_uint4(wh[i][0], wh[i][1], wh[i][2], wh[i][3]);
                *reinterpret_cast<uint4 *>(wop + kBox + off) = make_uint4(wl[i][0], wl[i][1], wl[i][2], wl[i][3]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();   // the operand tiles are in
            // ---- W^T = K^T (A diag(beta b))^T on the tensor cores, into the Gram's TMEM columns
            if (tid == 0) {
                ok = mbar_wait(&ctl->full, 1);
                if (ok) {
                    tc_fence_after();
                    constexpr uint32_t id_w = idesc_bf16_f32(128, 64, true, false);   // K^T MN-major
                    const uint32_t kb = smem_addr(smem + kPW), ab = smem_addr(wop);
                    // the lo products first: the accumulator rounds each instruction's sum
#pragma unroll
                    for (int hl = 1; hl >= 0; --hl)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_f16(tmem, smem_desc_sw128(kb + (uint32_t)ks * 2048u, kBox, 1024),
                                    smem_desc_sw128(ab + (uint32_t)hl * kBox + (uint32_t)ks * 32u, 0, 1024), id_w,
                                    (hl == 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(&ctl->mma);
            }
            ok = __syncthreads_and(ok && mbar_wait(&ctl->mma, 1));
            tc_fence_after();
            if (ok) {
                // ---- -W^T -> bf16 hi / lo tiles (row k = this thread's TMEM lane, tokens t
                // contiguous, 16-byte group c at position c ^ (k & 7)), staged in shared
                // memory over the dead keys and operand tiles, then one bulk copy to the record
                const int k = tid;
                uint8_t *wt = smem + kPWst;
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(cb * 32), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int c = cb * 4 + cc;
                        uint32_t hv[4], lv[4];
#pragma unroll
                        for (int p = 0; p < 4; ++p)
                            split_pair(-__uint_as_float(r[cc * 8 + 2 * p]), -__uint_as_float(r[cc * 8 + 2 * p + 1]),
                                       hv[p], lv[p]);
                        const int off = k * 128 + ((c ^ (k & 7)) << 4);
                        *reinterpret_cast<uint4 *>(wt + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                        *reinterpret_cast<uint4 *>(wt + 16384 + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
                    }
                }
                fence_async_smem();
                __syncthreads();
                if (tid == 0) {
                    bulk_store(rec + R::Wt, wt, 32768u);
                    bulk_commit();
                    bulk_wait_read_all();   // the staging area stays valid until the copy has read it
                }
            } else if (tid == 0 && a.d_err) {
                atomicExch(a.d_err, (int)HYPIC_ETIMEOUT);
            }
        }
    } else if (tid == 0 && a.d_err) {
        atomicExch(a.d_err, (int)HYPIC_ETIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

// ================================================================ pass 2: state

constexpr int kNS = 2;            // stages
// 23 warps: 0 TMA, 1-4 W/U operands, 5-20 state, 21 MMA issue, 22 a second MMA-issue
// warp (a single thread issues N = 64 products at about one per 60 cycles): without
// o_t it takes the second k half of Delta, with o_t the output products O1 and O2
template <bool O>
constexpr int state_threads() { return 736; }
constexpr int kWT = 128;          // W warps' threads
constexpr int kState = 512;       // state warps' threads

// stage: K (two 64-channel boxes), V (state half), Q (o_t), the head of the
// chunk's record (A tiles, gates); then, with o_t, one Gq buffer; then the -W^T
// operand tiles (two buffers without o_t, one with).
template <bool O>
struct Smem {
    static constexpr int K = 0, V = 2 * kBox, Q = 4 * kBox, Rec = (O ? 6 : 4) * kBox;
    static constexpr int Stage = Rec + ((hypic::Rec<O>::HeadBytes + 1023) / 1024) * 1024;
    static constexpr int NB = O ? 1 : 2;               // operand buffers
    static constexpr int Gqb = kNS * Stage;            // with o_t: Gq hi / lo (64 x 128 B each)
    static constexpr int Wt = Gqb + (O ? 16384 : 0);   // -W^T, per buffer hi / lo (128 rows x 128 B each)
    static constexpr int Ost = Wt + NB * 32768;        // with o_t: o staging, 8 tokens x 32 channels per state warp
    static constexpr int Ctl = Ost + (O ? 16 * 512 : 0);
};

// TMEM column map (512 allocated)
constexpr uint32_t kTx = 0;       // X^T half, fp32 (128 columns)
constexpr uint32_t kTxop = 128;   // X0^T operand: hi [128, 192), lo [192, 256), bf16 pairs;
                                  // with o_t then Delta^T hi / lo (O2 operand) in [128, 192)
constexpr uint32_t kTacc = 256;   // U^T - X0^T W^T, then Delta~^T operand in place (64)
constexpr uint32_t kTw = 320;     // W^T accumulator (64 columns)
constexpr uint32_t kTo1 = 384;    // O1^T accumulator (64 columns, o_t)
constexpr uint32_t kTo2 = 448;    // O2^T accumulator (64 columns, o_t)
constexpr uint32_t kTacc2 = 384;  // without o_t: the second k half of X0^T W^T (64 columns)

struct StateCtl {
    uint64_t full[kNS], empty[kNS];
    uint64_t wop_ready[2], wfree[2];                 // per operand buffer
    uint64_t gfull;                                  // o_t: Gq of the next chunk is in
    uint64_t xop_ready[2], dt_ready;                 // state warps -> MMA issuer
    uint64_t w_done, d_done, x_done;
    uint64_t o1_done, o2_done;                       // o_t: the output products of a chunk
    uint64_t o_free;                                 // o_t: the state warps have read O1, O2
    uint64_t drain[3];
    float redmax[16];
    float bo[kC];          // b_t of the chunk whose o_t is pending
    uint32_t tmem;
    int abort;
};
template <bool O>
constexpr int state_smem() { return Smem<O>::Ctl + (int)sizeof(StateCtl) + 1024; }
static_assert(state_smem<true>() <= 232448, "fits in one SM's shared memory");
static_assert(Smem<true>::Stage % 1024 == 0, "operand tiles 1024-byte aligned");

// max over the 16 state warps (named barrier 2)
__device__ __forceinline__ float state_max(float mx, StateCtl *ctl, int sw, int lane) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) ctl->redmax[sw] = mx;
    bar_sync(2, kState);
    mx = 0.f;
#pragma unroll
    for (int w = 0; w < 16; ++w) mx = fmaxf(mx, ctl->redmax[w]);
    bar_sync(2, kState);
    return mx;
}

// o_t = b_t O1 + O2 for this thread's 16 tokens (column group cg) of one chunk, as
// bf16 pairs (tokens 2q, 2q + 1 in opk[q]); then the warp arrives on `freed` (if
// given): O1 and O2 have been read
__device__ __forceinline__ void load_o(uint32_t to1, uint32_t to2, const float *b, float o2s, int cg, int lane,
                                       uint32_t (&opk)[8], uint64_t *freed) {
    uint32_t r1[16], r2[16];
    tmem_ld16(to1, r1);
    tmem_ld16(to2, r2);
    tmem_wait_ld();
    if (freed != nullptr) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(freed);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int t = cg * 16 + 2 * q;
        const __nv_bfloat162 v =
            __floats2bfloat162_rn(fmaf(b[t], __uint_as_float(r1[2 * q]), o2s * __uint_as_float(r2[2 * q])),
                                  fmaf(b[t + 1], __uint_as_float(r1[2 * q + 1]), o2s * __uint_as_float(r2[2 * q + 1])));
        opk[q] = *reinterpret_cast<const uint32_t *>(&v);
    }
}

// write those 16 tokens of channel quarter * 32 + lane, whose first token is row
// `crow` of [n_layers * N]: through the warp's staging tile, 8 tokens at a time,
// so that each lane stores one 16-byte run of 8 channels of one token
__device__ __forceinline__ void store_o(const ScanArgs &a, int h, int cg, int quarter, int lane, int64_t crow,
                                        int nvalid, const uint32_t (&opk)[8], __nv_bfloat16 *stg) {
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.o_out) + (int64_t)h * kD + quarter * 32 + (lane & 3) * 8;
    const int64_t rs = (int64_t)a.H * kD;   // elements from one token to the next
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

// 23 warps: six on some sub-partitions, 16384 / (6 x 32) registers -> at most 80 per thread
template <bool O>
__global__ void __maxnreg__(80)
    dense_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_q, const ScanArgs a, int64_t slots) {
    using R = Rec<O>;
    using SM = Smem<O>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align1024(smem_raw);
    StateCtl *ctl = reinterpret_cast<StateCtl *>(smem + SM::Ctl);
    volatile int *abortp = &ctl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int half = blockIdx.x & 1;   // 0: transition M, 1: state S
    // chains in the order of their segments, longest first (all layers and heads of
    // a segment together), so that the last wave holds the shortest chains
    const int unit = blockIdx.x >> 1;
    const int rank = unit / (a.H * a.n_layers);
    const int l = (unit / a.H) % a.n_layers;
    const int h = unit % a.H;
    const int seg = a.order ? a.order[rank] : rank;
    int64_t t0 = a.seg_offsets[seg], t1 = a.seg_offsets[seg + 1];
    const bool bad = !(t0 >= 0 && t0 <= t1 && t1 <= a.N);
    if (bad) t0 = t1 = 0;
    const int nc = (int)((t1 - t0 + kC - 1) / kC);
    const int64_t row0 = (int64_t)l * a.N + t0;
    const float *recs = a.ws + (((int64_t)l * a.H + h) * slots + seg + t0 / kC) * R::Floats;
    const bool with_o = O && half == 1;   // o_t comes from the state half
    const bool split_d = !with_o;         // the second issuer takes the second k half of Delta

    if (threadIdx.x == 0) {
        if (bad) flag_index_error(a.d_err);
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], with_o ? 2 : 1);   // with o_t both issuers read the stage
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->wop_ready[b], kWT / 32);
            mbar_init(&ctl->wfree[b], split_d ? 2 : 1);   // every issuer of Delta products commits
        }
        mbar_init(&ctl->xop_ready[0], kState / 32);
        mbar_init(&ctl->xop_ready[1], kState / 32);
        mbar_init(&ctl->dt_ready, kState / 32);
        mbar_init(&ctl->w_done, 1);
        mbar_init(&ctl->d_done, split_d ? 2 : 1);
        mbar_init(&ctl->x_done, 1);
        mbar_init(&ctl->o1_done, 1);
        mbar_init(&ctl->o2_done, 1);
        mbar_init(&ctl->o_free, kState / 32);
        for (int d = 0; d < 3; ++d) mbar_init(&ctl->drain[d], 1);
        mbar_init(&ctl->gfull, 1);
        ctl->abort = 0;
        mbar_fence_init();
        tma_prefetch(&tm_k);
        if (half) tma_prefetch(&tm_v);
        if (with_o) tma_prefetch(&tm_q);
    }
    if (warp == 0) tmem_alloc(&ctl->tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;

    constexpr uint32_t id_wu = idesc_bf16_f32(128, 64, true, false);    // K^T / V^T (MN-major) x A tiles
    constexpr uint32_t id_d = idesc_bf16_f32(128, 64, false, true);     // X0^T (TMEM) x W^T (MN-major)
    constexpr uint32_t id_x = idesc_bf16_f32(128, 128, false, true);    // Delta~^T (TMEM) x K (MN-major)
    constexpr uint32_t id_o = idesc_bf16_f32(128, 64, false, false);    // TMEM x Q / Gq (K-major)

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            for (int j = 0; j < nc; ++j) {
                const int s = j % kNS;
                if (!wait_or_abort(&ctl->empty[s], ((uint32_t)(j / kNS) & 1u) ^ 1u, abortp)) break;
                uint8_t *st = smem + s * SM::Stage;
                const int row = (int)(row0 + (int64_t)j * kC);
                // the transition half takes A diag(beta b) and the gates only
                const uint32_t rbytes = half ? (uint32_t)R::HeadBytes : 16384u + (uint32_t)(R::Head - R::G) * 4u;
                mbar_expect_tx(&ctl->full[s], (uint32_t)((2 + (half ? 2 : 0) + (with_o ? 2 : 0)) * kBox) + rbytes);
                tma_load_3d(st + SM::K, &tm_k, &ctl->full[s], 0, h, row);
                tma_load_3d(st + SM::K + kBox, &tm_k, &ctl->full[s], 64, h, row);
                if (half) {   // V only feeds the state half
                    tma_load_3d(st + SM::V, &tm_v, &ctl->full[s], 0, h, row);
                    tma_load_3d(st + SM::V + kBox, &tm_v, &ctl->full[s], 64, h, row);
                }
                if (with_o) {
                    tma_load_3d(st + SM::Q, &tm_q, &ctl->full[s], 0, h, row);
                    tma_load_3d(st + SM::Q + kBox, &tm_q, &ctl->full[s], 64, h, row);
                }
                const float *rj = recs + (int64_t)j * R::Floats;
                if (half) {
                    bulk_load(st + SM::Rec, rj, (uint32_t)R::HeadBytes, &ctl->full[s]);
                } else {
                    bulk_load(st + SM::Rec, rj, 16384u, &ctl->full[s]);
                    bulk_load(st + SM::Rec + R::G * 4, rj + R::G, (uint32_t)(R::Head - R::G) * 4u, &ctl->full[s]);
                }
                issued = j + 1;
            }
            if (*abortp)
                for (int j = issued - kNS < 0 ? 0 : issued - kNS; j < issued; ++j)
                    mbar_wait(&ctl->full[j % kNS], (uint32_t)(j / kNS) & 1u);
        } else if (lane == 1 && with_o) {
            // Gq of chunk j into its buffer once chunk j - 1's O2 products have read it
            // (o2_done of j cannot pass before this copy: O2 of j waits for it)
            int issued = 0;
            for (int j = 0; j < nc; ++j) {
                if (j > 0 && !wait_or_abort(&ctl->o2_done, (uint32_t)(j - 1) & 1u, abortp)) break;
                mbar_expect_tx(&ctl->gfull, 16384u);
                bulk_load(smem + SM::Gqb, recs + (int64_t)j * R::Floats + R::Gq, 16384u, &ctl->gfull);
                issued = j + 1;
            }
            if (*abortp && issued > 0) mbar_wait(&ctl->gfull, (uint32_t)(issued - 1) & 1u);
        }
    } else if (warp <= 4) {
        // ------------------------------------------------------------ W / U operand warps
        const int wt = threadIdx.x - 32;   // 0..127
        const bool issuer = wt == 0;
        const int quarter = warp & 3;
        for (int j = 0; j < nc; ++j) {
            const int s = j % kNS;
            const int b = j % SM::NB;
            const uint32_t use = (uint32_t)(j / SM::NB);
            uint8_t *st = smem + s * SM::Stage;
            const float *rec = reinterpret_cast<const float *>(st + SM::Rec);
            // the chunk is in, and the operand buffer's previous use is consumed
            bool ok = wait_or_abort(&ctl->full[s], (uint32_t)(j / kNS) & 1u, abortp);
            if (j >= SM::NB) ok = ok && wait_or_abort(&ctl->wfree[b], (use - 1u) & 1u, abortp);
            if (!bar_and(1, kWT, ok)) {
                *abortp = 1;
                break;
            }
            // ---- W^T = K^T (A diag(beta b))^T
            if (issuer) {
                tc_fence_after();
                const uint32_t kb = smem_addr(st + SM::K);
                const uint32_t ab2 = smem_addr(st + SM::Rec);
                const uint64_t dk0 = smem_desc_sw128(kb, kBox, 1024), da0 = smem_desc_sw128(ab2, 0, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t ad = dk0 + (uint64_t)(ks * 128);
                    mma_f16(tmem + kTw, ad, da0 + (uint64_t)(ks * 2), id_wu, ks > 0);
                    mma_f16(tmem + kTw, ad, da0 + (uint64_t)(512 + ks * 2), id_wu, 1u);
                }
                mma_commit(&ctl->w_done);
            }
            if (!bar_and(1, kWT, wait_or_abort(&ctl->w_done, (uint32_t)j & 1u, abortp))) {
                *abortp = 1;
                break;
            }
            tc_fence_after();
            // ---- -W^T -> bf16 hi / lo tiles, MN-major (row k, t contiguous, 128-byte swizzle)
            {
                const int k = quarter * 32 + lane;
                uint8_t *wtile = smem + SM::Wt + b * 32768;
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + kTw + (uint32_t)(cb * 32), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int c = cb * 4 + cc;
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int p = 0; p < 4; ++p)
                            split_pair(-__uint_as_float(r[cc * 8 + 2 * p]), -__uint_as_float(r[cc * 8 + 2 * p + 1]),
                                       hi[p], lo[p]);
                        const int off = k * 128 + ((c ^ (k & 7)) << 4);
                        *reinterpret_cast<uint4 *>(wtile + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4 *>(wtile + 16384 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
            }
            tc_fence_before();
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->wop_ready[b]);
        }
        if (issuer && *abortp) {   // drain: completes once this thread's MMAs are done
            mma_commit(&ctl->drain[0]);
            mbar_wait(&ctl->drain[0], 0);
        }
    } else if (warp < 21) {
        // ------------------------------------------------------------ state warps
        const int st = threadIdx.x - 160;           // 0..511
        const int sw = warp - 5;                    // 0..15
        const int cg = sw >> 2;                     // column group of this warp
        const int quarter = warp & 3;               // TMEM lanes this warp may touch
        const int m = quarter * 32 + lane;          // column of X = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        // this thread's X^T columns: k = p * 64 + cg * 16 .. +15 for the halves p = 0, 1,
        // converted half by half so the issuer can start on half 0 while half 1 converts
        const uint32_t tx0 = tmem + lane_off + kTx + (uint32_t)(cg * 16);
        const uint32_t txop = tmem + lane_off + kTxop + (uint32_t)(cg * 8);   // hi (+32: half 1; +64: lo)
        const uint32_t tdo = tmem + lane_off + kTxop + (uint32_t)(cg * 16);   // o_t: Delta^T hi / lo (tokens)
        const uint32_t tacc = tmem + lane_off + kTacc + (uint32_t)(cg * 16);
        const uint32_t to1 = tmem + lane_off + kTo1 + (uint32_t)(cg * 16);
        const uint32_t to2 = tmem + lane_off + kTo2 + (uint32_t)(cg * 16);
        __nv_bfloat16 *ostg = reinterpret_cast<__nv_bfloat16 *>(smem + SM::Ost) + sw * 256;   // o_t staging
        // Transition half: M_true = exp(lam_d + lam_exp ln2) M_stored, and each chunk
        // stores T_chunk M / b_C (log b_C into lam_d).  State half: S_true =
        // exp(ls) S_stored.  Either way the update only accumulates into TMEM; X is
        // rewritten only to renormalise (every 8 chunks for M, when ls < -20 for S)
        // or on a chunk whose total decay is below e^-40 (exact write-back form).
        int lam_exp = 0;
        double lam_d = 0.0;
        float ls = 0.f;
        // o_t: the previous chunk's O2 factor (1 / fD, or 1 where O2 took Delta itself) and
        // whether its Delta sits in the X0 operand columns (a chunk below e^-40)
        float o2s_prev = 1.f;
        bool steep_prev = false;

        {   // initial X^T: identity (transition) or zero (state)
            uint32_t r[16];
#pragma unroll
            for (int p = 0; p < 2; ++p) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    r[i] = __float_as_uint((half == 0 && p * 64 + cg * 16 + i == m) ? 1.f : 0.f);
                tmem_st16(tx0 + (uint32_t)(p * 64), r);
            }
            tmem_wait_st();
        }

        for (int j = 0; j < nc; ++j) {
            const int s = j % kNS;
            const uint8_t *stg = smem + s * SM::Stage;
            const float *rec = reinterpret_cast<const float *>(stg + SM::Rec);
            bool ok = wait_or_abort(&ctl->full[s], (uint32_t)(j / kNS) & 1u, abortp);
            // ---- scales of this chunk, from its record (while the previous update runs)
            const float LC = rec[R::LC];                // log of the chunk's total decay
            const bool slow = LC < -40.f;
            const bool renorm = slow || (half == 0 ? (j % 8 == 0) : (ls < -20.f));
            float g = 1.f;        // X_stored <- g * wscale * X_stored when rewritten
            float wscale = 1.f;
            float fP, fD;         // X0_true = fP * g * X_stored;  Delta~ = fD * (b_C / b) * Delta
            if (half == 0) {
                wscale = slow ? rec[R::BC] : 1.f;
                fP = 1.f;
                fD = slow ? 1.f : expf(-LC);
                if (!slow && st == 0) lam_d += (double)LC;   // only this thread writes lambda
            } else {
                if (slow) {
                    g = expf(ls);
                    wscale = rec[R::BC];
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
            if (j > 0) ok = ok && wait_or_abort(&ctl->x_done, (uint32_t)(j - 1) & 1u, abortp);
            // the previous chunk's O2 products read Delta from the X0 operand columns
            if (with_o && j > 0 && steep_prev) ok = ok && wait_or_abort(&ctl->o2_done, (uint32_t)(j - 1) & 1u, abortp);
            if (!bar_and(2, kState, ok)) {
                *abortp = 1;
                break;
            }
            tc_fence_after();
            if (half == 0 && renorm) {   // the transition's power-of-two renormalisation
                float mx = 0.f;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    uint32_t r[16];
                    tmem_ld16(tx0 + (uint32_t)(p * 64), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(__uint_as_float(r[i])));
                }
                const int e = exponent_of(state_max(mx, ctl, sw, lane));
                g = ldexpf(1.f, -e);
                lam_exp += e;
            }
            // ---- X round trip (TMEM only), per k half: operand X0_true (hi + lo), X_stored
            // rescaled if due; each half is announced as soon as it is in place
            {
                const float mult = g * fP, sc = g * wscale;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    uint32_t r[16], hi[8], lo[8];
                    tmem_ld16(tx0 + (uint32_t)(p * 64), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        split_pair(mult * __uint_as_float(r[2 * q]), mult * __uint_as_float(r[2 * q + 1]), hi[q],
                                   lo[q]);
                    tmem_st8(txop + (uint32_t)(p * 32), hi);
                    tmem_st8(txop + 64u + (uint32_t)(p * 32), lo);
                    if (renorm) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(sc * __uint_as_float(r[i]));
                        tmem_st16(tx0 + (uint32_t)(p * 64), r);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->xop_ready[p]);
                }
            }
            // ---- o_t of the previous chunk (its O1 and O2 complete), to memory while the
            // Delta products run; the O1 products of this chunk wait for o_free
            bool ok_o = true;
            if (with_o && j > 0) {
                ok_o = wait_or_abort(&ctl->o2_done, (uint32_t)(j - 1) & 1u, abortp);
                tc_fence_after();
                uint32_t opk[8];
                load_o(to1, to2, ctl->bo, o2s_prev, cg, lane, opk, &ctl->o_free);
                store_o(a, h, cg, quarter, lane, row0 + (int64_t)(j - 1) * kC, kC, opk, ostg);
            }
            // ---- Delta~^T = fD Delta^T diag(b_C / b) -> bf16 hi / lo in place
            // (with o_t also Delta^T itself, hi / lo, into the X0 operand columns, once
            // the O1 products have read X0 there)
            if (!bar_and(2, kState, ok_o && wait_or_abort(&ctl->d_done, (uint32_t)j & 1u, abortp) &&
                                        (!with_o || wait_or_abort(&ctl->o1_done, (uint32_t)j & 1u, abortp)))) {
                *abortp = 1;
                break;
            }
            tc_fence_after();
            {
                uint32_t r[16], hi[8], lo[8];
                tmem_ld16(tacc, r);
                if (split_d) {   // plus the second k half's accumulator
                    uint32_t r2[16];
                    tmem_ld16(tacc + (kTacc2 - kTacc), r2);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 16; ++q) r[q] = __float_as_uint(__uint_as_float(r[q]) + __uint_as_float(r2[q]));
                }
                tmem_wait_ld();
                if (with_o && slow) {   // O2 takes Delta itself (Delta~ may underflow)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        split_pair(__uint_as_float(r[2 * q]), __uint_as_float(r[2 * q + 1]), hi[q], lo[q]);
                    tmem_st8(tdo, hi);
                    tmem_st8(tdo + 8u, lo);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int t = cg * 16 + 2 * q;
                    split_pair(fD * rec[R::Gw + t] * __uint_as_float(r[2 * q]),
                               fD * rec[R::Gw + t + 1] * __uint_as_float(r[2 * q + 1]), hi[q], lo[q]);
                }
                tmem_st8(tacc, hi);          // tokens cg*16 .. +15: hi in the first 8 columns,
                tmem_st8(tacc + 8u, lo);     // lo in the next 8 (this thread's own columns)
                if (with_o && st < kC) ctl->bo[st] = rec[R::B + st];   // for this chunk's o store
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->dt_ready);
            o2s_prev = slow ? 1.f : 1.f / fD;
            steep_prev = slow;
        }

        // ------------------------------------------------------------ epilogue
        bool ok = true;
        if (nc > 0) ok = wait_or_abort(&ctl->x_done, (uint32_t)(nc - 1) & 1u, abortp);
        if (with_o && nc > 0) ok = ok && wait_or_abort(&ctl->o2_done, (uint32_t)(nc - 1) & 1u, abortp);
        if (bar_and(2, kState, ok)) {
            tc_fence_after();
            if (with_o && nc > 0) {
                uint32_t opk[8];
                load_o(to1, to2, ctl->bo, o2s_prev, cg, lane, opk, nullptr);
                store_o(a, h, cg, quarter, lane, row0 + (int64_t)(nc - 1) * kC,
                        (int)(t1 - t0 - (int64_t)(nc - 1) * kC), opk, ostg);
            }
            const int64_t u_out = ((int64_t)l * a.n_seg + seg) * a.H + h;
            uint32_t r[2][16];
            tmem_ld16(tx0, r[0]);
            tmem_ld16(tx0 + 64u, r[1]);
            tmem_wait_ld();
            float scale;
            if (half == 0) {
                float mx = 0.f;
#pragma unroll
                for (int p = 0; p < 2; ++p)
#pragma unroll
                    for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(__uint_as_float(r[p][i])));
                const int e = exponent_of(state_max(mx, ctl, sw, lane));
                scale = ldexpf(1.f, -e);
                lam_exp += e;
                if (st == 0) a.lam_out[u_out] = (float)(lam_d + (double)lam_exp * 0.69314718055994530942);
            } else {
                scale = expf(ls);
            }
            float *out = (half == 0 ? a.M_out : a.S_out) + u_out * kD * kD;
#pragma unroll
            for (int p = 0; p < 2; ++p)
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    out[(int64_t)(p * 64 + cg * 16 + i) * kD + m] = scale * __uint_as_float(r[p][i]);
        } else {
            *abortp = 1;
        }
    } else if (warp == 22 && split_d) {
        // ------------------------------------------------------------ second MMA issuer (no o_t
        // in this CTA): the second k half of X0^T W^T into its own accumulator
        if (lane == 0) {
            for (int j = 0; j < nc; ++j) {
                const int b = j % SM::NB;
                const uint32_t use = (uint32_t)(j / SM::NB);
                const uint32_t par = (uint32_t)j & 1u;
                // its accumulator has been read (Delta~ of the previous chunk is converted)
                if (j > 0 && !wait_or_abort(&ctl->x_done, par ^ 1u, abortp)) break;
                if (!wait_or_abort(&ctl->wop_ready[b], use & 1u, abortp)) break;
                if (!wait_or_abort(&ctl->xop_ready[1], par, abortp)) break;
                tc_fence_after();
                const uint32_t wtile = smem_addr(smem + SM::Wt + b * 32768);
            const uint64_t dwh = smem_desc_sw128(wtile, 16384, 1024);
#pragma unroll
                for (int kq = 0; kq < 4; ++kq) {
                    const int ks = 4 + kq;
                    const uint64_t bh = dwh + (uint64_t)(ks * 128);
                    const uint64_t bl = dwh + (uint64_t)(1024 + ks * 128);
                    const uint32_t ah = tmem + kTxop + (uint32_t)ks * 8u, al = ah + 64u;
                    mma_f16_ta(tmem + kTacc2, ah, bh, id_d, kq > 0 ? 1u : 0u);
                    mma_f16_ta(tmem + kTacc2, ah, bl, id_d, 1u);
                    mma_f16_ta(tmem + kTacc2, al, bh, id_d, 1u);
                }
                mma_commit(&ctl->d_done);
                mma_commit(&ctl->wfree[b]);
            }
            if (*abortp) {   // drain: completes once this thread's MMAs are done
                mma_commit(&ctl->drain[2]);
                mbar_wait(&ctl->drain[2], 0);
            }
        }
    } else if (warp == 22) {
        // ------------------------------------------------------------ output-product issuer (o_t):
        // O1^T = X0^T Q^T per k half as soon as that half of X0 is converted, then
        // O2^T = Delta^T Gq^T (three-term split) once Delta^T is in place
        if (lane == 0 && with_o) {
            for (int j = 0; j < nc; ++j) {
                const int s = j % kNS;
                const uint32_t par = (uint32_t)j & 1u;
                const uint8_t *stg = smem + s * SM::Stage;
                if (!wait_or_abort(&ctl->full[s], (uint32_t)(j / kNS) & 1u, abortp)) break;
                const uint32_t qb = smem_addr(stg + SM::Q);
                const uint64_t dq0 = smem_desc_sw128(qb, 0, 1024);
                // O2 reads Delta~ from its accumulator, or Delta from the X0 operand columns
                // on a chunk that decays below e^-40
                const bool steep = reinterpret_cast<const float *>(stg + SM::Rec)[R::LC] < -40.f;
                const uint32_t d2 = tmem + (steep ? kTxop : kTacc);
                bool ok = true;
                for (int p = 0; p < 2 && ok; ++p) {
                    ok = wait_or_abort(&ctl->xop_ready[p], par, abortp);
                    // O1 and O2 of the previous chunk have been read (store_o)
                    if (p == 0 && j > 0) ok = ok && wait_or_abort(&ctl->o_free, (uint32_t)(j - 1) & 1u, abortp);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kq = 0; kq < 4; ++kq) {
                        const int ks = p * 4 + kq;
                        const uint64_t bq = dq0 + (uint64_t)((ks >> 2) * (kBox >> 4) + (ks & 3) * 2);
                        const uint32_t ah = tmem + kTxop + (uint32_t)ks * 8u;
                        mma_f16_ta(tmem + kTo1, ah, bq, id_o, ks > 0);
                        mma_f16_ta(tmem + kTo1, ah + 64u, bq, id_o, 1u);
                    }
                }
                if (!ok) break;
                mma_commit(&ctl->o1_done);
                mma_commit(&ctl->empty[s]);   // its last read of the stage (Q)
                if (!wait_or_abort(&ctl->dt_ready, par, abortp)) break;
                if (!wait_or_abort(&ctl->gfull, par, abortp)) break;
                tc_fence_after();
                const uint32_t gq = smem_addr(smem + SM::Gqb);
                const uint64_t dg0 = smem_desc_sw128(gq, 0, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t gh = dg0 + (uint64_t)(ks * 2);
                    const uint64_t gl = dg0 + (uint64_t)(512 + ks * 2);
                    const uint32_t ah = d2 + (uint32_t)ks * 16u;
                    mma_f16_ta(tmem + kTo2, ah, gh, id_o, ks > 0);
                    mma_f16_ta(tmem + kTo2, ah, gl, id_o, 1u);
                    mma_f16_ta(tmem + kTo2, ah + 8u, gh, id_o, 1u);
                }
                mma_commit(&ctl->o2_done);
            }
            if (*abortp) {   // drain: completes once this thread's MMAs are done
                mma_commit(&ctl->drain[2]);
                mbar_wait(&ctl->drain[2], 0);
            }
        }
    } else if (lane == 0) {
        // ------------------------------------------------------------ MMA issuer (warp 21)
        for (int j = 0; j < nc; ++j) {
            const int s = j % kNS;
            const int b = j % SM::NB;
            const uint32_t use = (uint32_t)(j / SM::NB);
            const uint32_t par = (uint32_t)j & 1u;
            const uint8_t *stg = smem + s * SM::Stage;
            // the accumulator is free (the previous update and, with o_t, the previous O2
            // products have read Delta~), the chunk is in
            if (j > 0 && !wait_or_abort(&ctl->x_done, par ^ 1u, abortp)) break;
            if (with_o && j > 0 && !wait_or_abort(&ctl->o2_done, par ^ 1u, abortp)) break;
            if (!wait_or_abort(&ctl->full[s], (uint32_t)(j / kNS) & 1u, abortp)) break;
            // ---- U^T = V^T (A diag(beta))^T into the accumulator (state half)
            if (half) {
                tc_fence_after();
                const uint32_t vb = smem_addr(stg + SM::V), ab = smem_addr(stg + SM::Rec + R::Ab * 4);
                const uint64_t dv0 = smem_desc_sw128(vb, kBox, 1024), dab0 = smem_desc_sw128(ab, 0, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t ad = dv0 + (uint64_t)(ks * 128);
                    mma_f16(tmem + kTacc, ad, dab0 + (uint64_t)(ks * 2), id_wu, ks > 0);
                    mma_f16(tmem + kTacc, ad, dab0 + (uint64_t)(512 + ks * 2), id_wu, 1u);
                }
            }
            // ---- Delta^T = U^T - X0^T W^T (three-term split), per k half
            if (!wait_or_abort(&ctl->wop_ready[b], use & 1u, abortp)) break;
            const uint32_t wtile = smem_addr(smem + SM::Wt + b * 32768);
            const uint64_t dwh = smem_desc_sw128(wtile, 16384, 1024);
            bool ok = true;
            for (int p = 0; p < (split_d ? 1 : 2) && ok; ++p) {   // split: the second half is warp 22's
                ok = wait_or_abort(&ctl->xop_ready[p], par, abortp);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kq = 0; kq < 4; ++kq) {
                    const int ks = p * 4 + kq;
                    const uint64_t bh = dwh + (uint64_t)(ks * 128);
                    const uint64_t bl = dwh + (uint64_t)(1024 + ks * 128);
                    const uint32_t ah = tmem + kTxop + (uint32_t)ks * 8u, al = ah + 64u;
                    mma_f16_ta(tmem + kTacc, ah, bh, id_d, (half || ks > 0) ? 1u : 0u);
                    mma_f16_ta(tmem + kTacc, ah, bl, id_d, 1u);
                    mma_f16_ta(tmem + kTacc, al, bh, id_d, 1u);
                }
            }
            if (!ok) break;
            mma_commit(&ctl->d_done);
            mma_commit(&ctl->wfree[b]);
            // ---- X^T += Delta~^T K (K as the MN-major B operand: row t, channels contiguous)
            if (!wait_or_abort(&ctl->dt_ready, par, abortp)) break;
            tc_fence_after();
            const uint32_t kb = smem_addr(stg + SM::K);
            const uint64_t dkb = smem_desc_sw128(kb, kBox, 1024);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t bd = dkb + (uint64_t)(ks * 128);
                const uint32_t ah = tmem + kTacc + (uint32_t)ks * 16u;
                mma_f16_ta(tmem + kTx, ah, bd, id_x, 1u);
                mma_f16_ta(tmem + kTx, ah + 8u, bd, id_x, 1u);
            }
            mma_commit(&ctl->x_done);
            mma_commit(&ctl->empty[s]);   // its last read of the stage (K; with o_t the other issuer reads Q)
        }
        if (*abortp) {   // drain: completes once this thread's MMAs are done
            mma_commit(&ctl->drain[1]);
            mbar_wait(&ctl->drain[1], 0);
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

// ================================================================ pass 2 without o_t: both halves
//
// One CTA per chain holds X^T = [M | S]^T whole (two 128-column halves in TMEM) and
// walks its chunks with the two halves interleaved, so that one half's CUDA-core
// conversions overlap the other half's tensor products.  -W^T comes ready from
// the record (the preparation pass built it), so both halves read one copy.
// Each half has its own X0 operand: hi in TMEM, lo in shared memory (TMEM holds
// X, X0 hi and Delta of both halves: 2 x (128 + 64 + 64) columns).  Each half has
// its own group of eight conversion warps, which per chunk j run
//   X0(j) | Delta~(j)
// while that half's issuing thread runs
//   [U^T ->] Delta^T = U^T - X0^T W^T (three-term split) | X^T += Delta~^T K,
// so the halves' pipelines advance independently on one tensor pipe.
// 19 warps: 0 TMA, 1 issuer for M, 2 issuer for S, 3-10 conversions for M,
// 11-18 conversions for S.  A launch whose last wave would fill at most half the
// SMs runs that wave's chains as single halves, one CTA each (the other half's
// issuer and conversion warps stay idle), so the wave spreads over twice the SMs.

constexpr int kPairThreads = 608;
struct PairSmem {
    static constexpr int K = 0, V = 2 * kBox, Tiles = 4 * kBox;          // per stage
    static constexpr int TileBytes = hypic::Rec<false>::G * 4;           // -W^T and A diag(beta) tiles
    static constexpr int Stage = Tiles + TileBytes;
    static constexpr int X0lo = kNS * Stage;                             // per half: 2 k halves x 16 KB
    static constexpr int Ctl = X0lo + 2 * 32768;
};
// TMEM, per half x at 256 x: X^T (fp32, 128 columns), X0^T hi (bf16 pairs, 64),
// Delta^T accumulator then Delta~^T hi / lo in place (64)
__device__ __forceinline__ uint32_t kPX(int x) { return (uint32_t)x * 256u; }
__device__ __forceinline__ uint32_t kPXh(int x) { return (uint32_t)x * 256u + 128u; }
__device__ __forceinline__ uint32_t kPD(int x) { return (uint32_t)x * 256u + 192u; }

struct PairCtl {
    uint64_t full[kNS], empty[kNS];
    uint64_t xop_ready[2][2];   // [half][k half] the half's X0 operand is in place
    uint64_t dt_ready[2][4];    // [half][16-token block] the half's Delta~ block is in place
    uint64_t d_done[2];         // the half's Delta products are done
    uint64_t x_done[2];         // the half's update is done
    uint64_t drain[2];
    float gates[kNS][hypic::Rec<false>::GateFloats];   // b_C / b, log b_C, b_C of the staged chunk
    float redmax[16];
    uint32_t tmem;
    int abort;
};
constexpr int pair_smem() { return PairSmem::Ctl + (int)sizeof(PairCtl) + 1024; }
static_assert(pair_smem() <= 232448, "fits in one SM's shared memory");
static_assert(PairSmem::Stage % 1024 == 0 && PairSmem::Tiles % 1024 == 0 && PairSmem::X0lo % 1024 == 0,
              "operand tiles 1024-byte aligned");
static_assert((hypic::Rec<false>::GateFloats * 4) % 16 == 0, "gate copy in 16-byte units");

// max over the 8 warps of one half's group (named barrier 2 + half)
__device__ __forceinline__ float group_max(float mx, PairCtl *ctl, int x, int gw, int lane) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) ctl->redmax[x * 8 + gw] = mx;
    bar_sync(2 + x, kState / 2);
    mx = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) mx = fmaxf(mx, ctl->redmax[x * 8 + w]);
    bar_sync(2 + x, kState / 2);
    return mx;
}

// X0 operand of one half: this thread's 32 rows k (two 16-row groups) of its column m
// of X in each k half, times `mult`, split into bf16 hi (TMEM, A operand) and lo
// (shared memory, K-major row m, 128-byte swizzle); X rewritten times `sc` when
// `rewrite`; each k half announced as soon as it is in place.  One TMEM load per
// k half (32 columns), so the first k half is ready after one load round trip.
__device__ __forceinline__ void pair_x0(uint32_t tx, uint32_t txh, uint8_t *lo_tile, int m, int sub, float mult,
                                       float sc, bool rewrite, uint64_t *ready, int lane) {
    const uint64_t mult2 = pk2(mult, mult);
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        uint32_t r[32], hi[16], lo[16];
        tmem_ld32(tx + (uint32_t)(p * 64 + sub * 32), r);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            float x0, x1;
            upk2(mul2(mult2, pk2(__uint_as_float(r[2 * q]), __uint_as_float(r[2 * q + 1]))), x0, x1);
            split_pair(x0, x1, hi[q], lo[q]);
        }
        tmem_st16(txh + (uint32_t)(p * 32 + sub * 16), hi);
        uint8_t *row = lo_tile + p * 16384 + m * 128;
#pragma unroll
        for (int g = 0; g < 4; ++g)   // this thread's four 16-byte groups of the row
            *reinterpret_cast<uint4 *>(row + (((4 * sub + g) ^ (m & 7)) << 4)) =
                make_uint4(lo[4 * g], lo[4 * g + 1], lo[4 * g + 2], lo[4 * g + 3]);
        if (rewrite) {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(sc * __uint_as_float(r[i]));
            tmem_st32(tx + (uint32_t)(p * 64 + sub * 32), r);
        }
        tmem_wait_st();
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ready[p]);
    }
}

// Delta~^T = fD Delta^T diag(b_C / b) in place, this thread's 32 tokens (16-token
// blocks 2 sub and 2 sub + 1, one TMEM load), bf16 hi / lo; each block announced
// as soon as it is in place
__device__ __forceinline__ void pair_dt(uint32_t tacc, float fD, const float *gw, int sub, int lane,
                                        uint64_t *ready) {
    uint32_t r[32];
    tmem_ld32(tacc + (uint32_t)(sub * 32), r);
    tmem_wait_ld();
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
        const int cg = sub * 2 + c2;
        const float4 *g4 = reinterpret_cast<const float4 *>(gw + cg * 16);
        float sc[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 gv = g4[i];
            sc[4 * i] = fD * gv.x;
            sc[4 * i + 1] = fD * gv.y;
            sc[4 * i + 2] = fD * gv.z;
            sc[4 * i + 3] = fD * gv.w;
        }
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float x0, x1;
            upk2(mul2(pk2(sc[2 * q], sc[2 * q + 1]),
                      pk2(__uint_as_float(r[c2 * 16 + 2 * q]), __uint_as_float(r[c2 * 16 + 2 * q + 1]))),
                 x0, x1);
            split_pair(x0, x1, hi[q], lo[q]);
        }
        tmem_st8(tacc + (uint32_t)(cg * 16), hi);
        tmem_st8(tacc + (uint32_t)(cg * 16 + 8), lo);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ready[cg]);
    }
}

// Scale bookkeeping of one half for one chunk (as the two-CTA form).  Transition
// (h = 0): M_true = exp(lam_d + lam_exp ln2) M_stored, each chunk stores T_chunk M /
// b_C; state (h = 1): S_true = exp(ls) S_stored.  The update only accumulates; X
// is rewritten to renormalise (M every 8 chunks, S when ls < -20) or on a chunk
// whose decay is below e^-40 (exact write-back form).
struct HalfScale {
    float g, wscale, fP, fD;
    bool renorm, slow;
};

__device__ __forceinline__ HalfScale pair_scale(int h, int j, const float *gates, float &ls, double &lam_d,
                                                bool writer) {
    using R = Rec<false>;
    HalfScale z;
    const float LC = gates[R::LC - R::G];
    z.slow = LC < -40.f;
    z.renorm = z.slow || (h == 0 ? (j % 8 == 0) : (ls < -20.f));
    z.g = 1.f;
    z.wscale = 1.f;
    if (h == 0) {
        z.wscale = z.slow ? gates[R::BC - R::G] : 1.f;
        z.fP = 1.f;
        z.fD = z.slow ? 1.f : expf(-LC);
        if (!z.slow && writer) lam_d += (double)LC;
    } else if (z.slow) {
        z.g = expf(ls);
        z.wscale = gates[R::BC - R::G];
        z.fP = 1.f;
        z.fD = 1.f;
        ls = 0.f;
    } else {
        if (z.renorm) {
            const int q = (int)rintf(ls * 1.44269504088896341f);
            z.g = ldexpf(1.f, q);
            ls -= (float)q * 0.69314718055994531f;
        }
        z.fP = expf(ls);
        z.fD = expf(-(ls + LC));
        ls += LC;
    }
    return z;
}

__global__ void __launch_bounds__(kPairThreads, 1)
    dense_pair_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const ScanArgs a, int64_t slots, int n_pair) {
    using R = Rec<false>;
    using SM = PairSmem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align1024(smem_raw);
    PairCtl *ctl = reinterpret_cast<PairCtl *>(smem + SM::Ctl);
    volatile int *abortp = &ctl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // chains in the order of their segments, longest first (all layers and heads of
    // a segment together), so that the last wave holds the shortest chains.  CTAs
    // [0, n_pair) run both halves of chain blockIdx.x; each CTA after them runs one
    // half of one of the remaining chains (a last wave shorter than half the SMs is
    // spread over twice as many SMs)
    const bool split = (int)blockIdx.x >= n_pair;
    const int unit = split ? n_pair + (((int)blockIdx.x - n_pair) >> 1) : (int)blockIdx.x;
    const int only = split ? (((int)blockIdx.x - n_pair) & 1) : -1;   // the one half run here, or -1
    const int rank = unit / (a.H * a.n_layers);
    const int l = (unit / a.H) % a.n_layers;
    const int h = unit % a.H;
    const int seg = a.order ? a.order[rank] : rank;
    int64_t t0 = a.seg_offsets[seg], t1 = a.seg_offsets[seg + 1];
    const bool bad = !(t0 >= 0 && t0 <= t1 && t1 <= a.N);
    if (bad) t0 = t1 = 0;
    const int nc = (int)((t1 - t0 + kC - 1) / kC);
    const int64_t row0 = (int64_t)l * a.N + t0;
    const float *recs = a.ws + (((int64_t)l * a.H + h) * slots + seg + t0 / kC) * R::Floats;

    if (threadIdx.x == 0) {
        if (bad) flag_index_error(a.d_err);
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], split ? 1 : 2);   // the issuers' updates read the stage last
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&ctl->xop_ready[x][0], kState / 64);   // the half's 8 conversion warps
            mbar_init(&ctl->xop_ready[x][1], kState / 64);
            for (int q = 0; q < 4; ++q) mbar_init(&ctl->dt_ready[x][q], 4);   // the 4 warps converting block q
            mbar_init(&ctl->d_done[x], 1);
            mbar_init(&ctl->x_done[x], 1);
            mbar_init(&ctl->drain[x], 1);
        }
        ctl->abort = 0;
        mbar_fence_init();
        tma_prefetch(&tm_k);
        tma_prefetch(&tm_v);
    }
    if (warp == 0) tmem_alloc(&ctl->tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;

    constexpr uint32_t id_wu = idesc_bf16_f32(128, 64, true, false);    // V^T (MN-major) x A tiles
    constexpr uint32_t id_d = idesc_bf16_f32(128, 64, false, true);     // X0^T (K-major) x W^T (MN-major)
    constexpr uint32_t id_x = idesc_bf16_f32(128, 128, false, true);    // Delta~^T (TMEM) x K (MN-major)

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            for (int j = 0; j < nc; ++j) {
                const int s = j % kNS;
                if (!wait_or_abort(&ctl->empty[s], ((uint32_t)(j / kNS) & 1u) ^ 1u, abortp)) break;
                uint8_t *st = smem + s * SM::Stage;
                const int row = (int)(row0 + (int64_t)j * kC);
                const float *rj = recs + (int64_t)j * R::Floats;
                mbar_expect_tx(&ctl->full[s], (uint32_t)(4 * kBox + SM::TileBytes + R::GateFloats * 4));
                tma_load_3d(st + SM::K, &tm_k, &ctl->full[s], 0, h, row);
                tma_load_3d(st + SM::K + kBox, &tm_k, &ctl->full[s], 64, h, row);
                tma_load_3d(st + SM::V, &tm_v, &ctl->full[s], 0, h, row);
                tma_load_3d(st + SM::V + kBox, &tm_v, &ctl->full[s], 64, h, row);
                bulk_load(st + SM::Tiles, rj, (uint32_t)SM::TileBytes, &ctl->full[s]);
                bulk_load(ctl->gates[s], rj + R::G, (uint32_t)(R::GateFloats * 4), &ctl->full[s]);
                issued = j + 1;
            }
            if (*abortp)
                for (int j = issued - kNS < 0 ? 0 : issued - kNS; j < issued; ++j)
                    mbar_wait(&ctl->full[j % kNS], (uint32_t)(j / kNS) & 1u);
        }
    } else if (warp <= 2) {
        // ------------------------------------------------------------ MMA issuers: warp 1 the
        // transition half, warp 2 the state half
        if (lane == 0 && (only < 0 || only == warp - 1)) {
            const int x = warp - 1;
            const uint32_t dacc = tmem + kPD(x), xh = tmem + kPXh(x);
            const uint32_t acc0 = x == 1 ? 1u : 0u;   // the state half adds to U^T
            // shared-memory descriptors, built once per stage: an operand offset of o bytes
            // adds o >> 4 to the start-address field (no carry: addresses < 256 KB)
            uint64_t d_wh[kNS], d_wl[kNS], d_k[kNS], d_v[kNS], d_a[kNS];
#pragma unroll
            for (int s = 0; s < kNS; ++s) {
                const uint32_t tb = smem_addr(smem + s * SM::Stage + SM::Tiles);
                d_wh[s] = smem_desc_sw128(tb + (uint32_t)R::Wt * 4u, 16384, 1024);
                d_wl[s] = smem_desc_sw128(tb + (uint32_t)R::Wt * 4u + 16384u, 16384, 1024);
                d_k[s] = smem_desc_sw128(smem_addr(smem + s * SM::Stage + SM::K), kBox, 1024);
                d_v[s] = smem_desc_sw128(smem_addr(smem + s * SM::Stage + SM::V), kBox, 1024);
                d_a[s] = smem_desc_sw128(tb + (uint32_t)R::Ab * 4u, 0, 1024);
            }
            const uint64_t d_lo = smem_desc_sw128(smem_addr(smem + SM::X0lo + x * 32768), 0, 1024);
            for (int j = 0; j < nc; ++j) {
                const int s = j % kNS;
                const uint32_t par = (uint32_t)j & 1u;
                const uint64_t wh = s ? d_wh[1] : d_wh[0], wl = s ? d_wl[1] : d_wl[0];
                // the accumulator is free (the previous update has read Delta~), the chunk is in
                if (j > 0 && !wait_or_abort(&ctl->x_done[x], par ^ 1u, abortp)) break;
                if (!wait_or_abort(&ctl->full[s], (uint32_t)(j / kNS) & 1u, abortp)) break;
                // ---- U^T = V^T (A diag(beta))^T into the accumulator (state half), lo first
                if (x == 1) {
                    tc_fence_after();
                    const uint64_t vd = s ? d_v[1] : d_v[0], ad = s ? d_a[1] : d_a[0];
#pragma unroll
                    for (int hl = 1; hl >= 0; --hl)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_f16(dacc, vd + (uint64_t)(ks * 128), ad + (uint64_t)(hl * 512 + ks * 2), id_wu,
                                    (hl == 0 || ks > 0) ? 1u : 0u);
                }
                // ---- Delta^T = U^T - X0^T W^T (three-term split), per k half: hi x lo and
                // lo x hi first, then hi x hi (the accumulator rounds each instruction's sum)
                bool ok = true;
                for (int p = 0; p < 2 && ok; ++p) {
                    ok = wait_or_abort(&ctl->xop_ready[x][p], par, abortp);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kq = 0; kq < 4; ++kq) {
                        const int ks = p * 4 + kq;
                        mma_f16_ta(dacc, xh + (uint32_t)ks * 8u, wl + (uint64_t)(ks * 128), id_d,
                                   (p > 0 || kq > 0) ? 1u : acc0);
                        mma_f16(dacc, d_lo + (uint64_t)(p * 1024 + kq * 2), wh + (uint64_t)(ks * 128), id_d, 1u);
                    }
#pragma unroll
                    for (int kq = 0; kq < 4; ++kq) {
                        const int ks = p * 4 + kq;
                        mma_f16_ta(dacc, xh + (uint32_t)ks * 8u, wh + (uint64_t)(ks * 128), id_d, 1u);
                    }
                }
                if (!ok) break;
                mma_commit(&ctl->d_done[x]);
                // ---- X^T += Delta~^T K (K as the MN-major B operand: row t, channels contiguous),
                // each 16-token block as soon as its Delta~ is converted (lo, then hi)
                const uint64_t kd = s ? d_k[1] : d_k[0];
                for (int ks = 0; ks < 4 && ok; ++ks) {
                    ok = wait_or_abort(&ctl->dt_ready[x][ks], par, abortp);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int hl = 1; hl >= 0; --hl)
                        mma_f16_ta(tmem + kPX(x), dacc + (uint32_t)ks * 16u + (uint32_t)hl * 8u,
                                   kd + (uint64_t)(ks * 128), id_x, 1u);
                }
                if (!ok) break;
                mma_commit(&ctl->x_done[x]);
                mma_commit(&ctl->empty[s]);
            }
            if (*abortp) {   // drain: completes once this thread's MMAs are done
                mma_commit(&ctl->drain[x]);
                mbar_wait(&ctl->drain[x], 0);
            }
        }
    } else if (only < 0 || ((warp - 3) >> 3) == only) {
        // ------------------------------------------------------------ conversion warps: warps
        // 3..10 take the transition half, warps 11..18 the state half, each group its own
        // pipeline (named barrier 2 + half) with two 16-column groups a thread, so that one
        // half's conversions run while the other half's products do
        const int st = threadIdx.x - 96;            // 0..511
        const int sw = warp - 3;                    // 0..15
        const int x = sw >> 3;                      // this group's half
        const int gt = st & 255;                    // thread within the group
        const int sub = (sw >> 2) & 1;              // column groups 2 sub and 2 sub + 1
        const int quarter = warp & 3;               // TMEM lanes this warp may touch
        const int m = quarter * 32 + lane;          // column of X = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int gbar = 2 + x;
        int lam_exp = 0;
        double lam_d = 0.0;
        float ls = 0.f;

        {   // initial X^T of this half: identity (transition) or zero (state)
            uint32_t r[16];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int cg = sub * 2 + c2;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        r[i] = __float_as_uint((x == 0 && p * 64 + cg * 16 + i == m) ? 1.f : 0.f);
                    tmem_st16(tmem + lane_off + kPX(x) + (uint32_t)(p * 64 + cg * 16), r);
                }
            tmem_wait_st();
        }

        bool alive = true;
        for (int j = 0; j < nc && alive; ++j) {
            const int s = j % kNS;
            const uint32_t par = (uint32_t)j & 1u;
            const float *gates = ctl->gates[s];
            // ---- the chunk's scales as soon as its gates are in (register work, kept off
            // the wait for the previous update); then X0 of this half once that update is done
            bool ok = wait_or_abort(&ctl->full[s], (uint32_t)(j / kNS) & 1u, abortp);
            const HalfScale z = pair_scale(x, j, gates, ls, lam_d, gt == 0);
            if (j > 0) ok = ok && wait_or_abort(&ctl->x_done[x], par ^ 1u, abortp);
            if (!bar_and(gbar, kState / 2, ok)) {
                alive = false;
                break;
            }
            tc_fence_after();
            float g = z.g;
            if (x == 0 && z.renorm) {   // the transition's power-of-two renormalisation
                float mx = 0.f;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_off + kPX(0) + (uint32_t)(p * 64 + sub * 32), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(__uint_as_float(r[i])));
                }
                const int e = exponent_of(group_max(mx, ctl, x, sw & 7, lane));
                g = ldexpf(1.f, -e);
                lam_exp += e;
            }
            pair_x0(tmem + lane_off + kPX(x), tmem + lane_off + kPXh(x), smem + SM::X0lo + x * 32768, m, sub,
                    g * z.fP, g * z.wscale, z.renorm, ctl->xop_ready[x], lane);
            // ---- Delta~ of this half, once its Delta products are done
            if (!bar_and(gbar, kState / 2, wait_or_abort(&ctl->d_done[x], par, abortp))) {
                alive = false;
                break;
            }
            tc_fence_after();
            pair_dt(tmem + lane_off + kPD(x), z.fD, gates + (R::Gw - R::G), sub, lane, ctl->dt_ready[x]);
        }

        // ------------------------------------------------------------ epilogue: this half
        bool ok = alive;
        if (ok && nc > 0) ok = wait_or_abort(&ctl->x_done[x], (uint32_t)(nc - 1) & 1u, abortp);
        if (bar_and(gbar, kState / 2, ok)) {
            tc_fence_after();
            const int64_t u_out = ((int64_t)l * a.n_seg + seg) * a.H + h;
            uint32_t r[2][2][16];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                for (int p = 0; p < 2; ++p)
                    tmem_ld16(tmem + lane_off + kPX(x) + (uint32_t)(p * 64 + (sub * 2 + c2) * 16), r[c2][p]);
            tmem_wait_ld();
            float scale;
            if (x == 0) {
                float mx = 0.f;
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                    for (int p = 0; p < 2; ++p)
#pragma unroll
                        for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(__uint_as_float(r[c2][p][i])));
                const int e = exponent_of(group_max(mx, ctl, x, sw & 7, lane));
                scale = ldexpf(1.f, -e);
                lam_exp += e;
                if (gt == 0) a.lam_out[u_out] = (float)(lam_d + (double)lam_exp * 0.69314718055994530942);
            } else {
                scale = expf(ls);
            }
            float *out = (x == 0 ? a.M_out : a.S_out) + u_out * kD * kD;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                for (int p = 0; p < 2; ++p)
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        out[(int64_t)(p * 64 + (sub * 2 + c2) * 16 + i) * kD + m] = scale * __uint_as_float(r[c2][p][i]);
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

// ================================================================ longest first

constexpr int kLptMax = 4096;   // segments ranked; beyond this the given order is kept

// order[rank] = segment, by length descending (ties: lower index first); a segment
// with bad offsets counts as empty.  One CTA.
__global__ void __launch_bounds__(1024) lpt_order_kernel(const int64_t *seg_offsets, int n_seg, int64_t N,
                                                         int *order) {
    __shared__ int64_t len[kLptMax];
    const bool rank = n_seg <= kLptMax;
    for (int i = threadIdx.x; i < n_seg && rank; i += blockDim.x) {
        const int64_t t0 = seg_offsets[i], t1 = seg_offsets[i + 1];
        len[i] = (t0 >= 0 && t0 <= t1 && t1 <= N) ? t1 - t0 : 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n_seg; i += blockDim.x) {
        if (!rank) {
            order[i] = i;
            continue;
        }
        const int64_t li = len[i];
        int r = 0;
        for (int j = 0; j < n_seg; ++j) r += (len[j] > li) || (len[j] == li && j < i);
        order[r] = i;
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    return n;
}

// bytes of the records (then the order array, 256-byte aligned)
int64_t records_bytes(const ScanArgs &a) {
    const int64_t b = (int64_t)a.n_layers * a.H * n_slots(a.N, a.n_seg) * (a.o_out ? Rec<true>::Bytes : Rec<false>::Bytes);
    return (b + 255) / 256 * 256;
}

template <bool O>
cudaError_t launch_two_pass(const ScanArgs &a0, cudaStream_t s) {
    ScanArgs a = a0;
    if (a.n_seg > 1) {   // rank the segments (one segment: nothing to order)
        int *order = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(a0.ws) + records_bytes(a0));
        lpt_order_kernel<<<1, 1024, 0, s>>>(a.seg_offsets, a.n_seg, a.N, order);
        cudaError_t e0 = cudaGetLastError();
        if (e0 != cudaSuccess) return e0;
        a.order = order;
    }
    const int64_t units = (int64_t)a.n_layers * a.n_seg * a.H;
    const uint64_t rows = (uint64_t)a.n_layers * (uint64_t)a.N;
    CUtensorMap mk, mv, mq;
    if (!make_tensor_map_3d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k, 128, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v, 128, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, O ? a.q : a.k, 128, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int64_t slots = n_slots(a.N, a.n_seg);
    cudaError_t e = cudaFuncSetAttribute(dense_prep_kernel<O>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
    if (e != cudaSuccess) return e;
    dense_prep_kernel<O><<<dim3((unsigned)(slots * a.H), (unsigned)a.n_layers), kPThreads, kPSmem, s>>>(mk, mq, a,
                                                                                                     slots);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (O) {
        e = cudaFuncSetAttribute(dense_state_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 state_smem<true>());
        if (e != cudaSuccess) return e;
        dense_state_kernel<true><<<(unsigned)(2 * units), state_threads<true>(), state_smem<true>(), s>>>(mk, mv, mq,
                                                                                                      a, slots);
    } else {
        e = cudaFuncSetAttribute(dense_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem());
        if (e != cudaSuccess) return e;
        // one CTA per SM: a last wave of at most half the SMs runs its chains' halves
        // on separate SMs (a lone half steps faster than an interleaved pair)
        const int64_t sms = sm_count(), tail = units % sms;
        const int64_t n_pair = (tail > 0 && 2 * tail <= sms) ? units - tail : units;
        dense_pair_kernel<<<(unsigned)(2 * units - n_pair), kPairThreads, pair_smem(), s>>>(mk, mv, a, slots,
                                                                                             (int)n_pair);
    }
    return cudaGetLastError();
}

}  // namespace

// ---------------------------------------------------------------- host side

bool scan_dense_ws_shape(const ScanArgs &a) {
    return a.fam == HYPIC_DENSE && a.in_dtype == HYPIC_BF16 && a.dk == 128 && a.dv == 128 && a.N > 0 &&
           (int64_t)a.n_layers * a.N < ((int64_t)1 << 31) &&
           (int64_t)a.n_layers * a.n_seg * a.H < ((int64_t)1 << 30) &&
           n_slots(a.N, a.n_seg) * a.H < ((int64_t)1 << 31) && a.n_layers <= 65535;
}

bool scan_dense_ws_supported(const ScanArgs &a) {
    return scan_dense_ws_shape(a) && tensor_map_encoder() != nullptr;
}

int64_t scan_dense_ws_bytes(const ScanArgs &a) {
    return records_bytes(a) + ((int64_t)a.n_seg * 4 + 255) / 256 * 256;
}

cudaError_t launch_scan_dense_ws(const ScanArgs &a, cudaStream_t s) {
    if ((int64_t)a.n_layers * a.n_seg * a.H == 0) return cudaSuccess;
    return a.o_out ? launch_two_pass<true>(a, s) : launch_two_pass<false>(a, s);
}

}  // namespace hypic
