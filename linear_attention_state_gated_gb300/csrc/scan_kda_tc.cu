// scan_kda_tc.cu -- segment scan of the KDA-style family (a gate per key channel
// inside the erasing update, T_t = diag(alpha_t)(I - beta_t k_t k_t^T)) on tcgen05
// tensor cores, bf16 k / v, d_k = d_v = 128, no o_t.
//
// Two passes.  The pair of a concatenation is the composition of the pairs of its
// parts, T(C1.C2) = T(C2) T(C1) and S(C1.C2|0) = T(C2) S(C1|0) + S(C2|0), so:
//   1. every chunk of 64 tokens of every segment becomes a cached pair (lambda_c,
//      M_c, S_c) with T_c = exp(lambda_c) M_c, all chunks independently
//      (scan_kda_chunk_kernel: one persistent CTA per SM walks the chunks, loading
//      the next chunk's tiles while the current one's products and epilogues run);
//   2. each segment folds its chunks' pairs in order with the composed-prefix
//      kernels (the state's chain from zero and the operator chain from I).
//
// The chunk's pair in closed form (WY / UT form of the per-channel gated delta
// rule).  Inside a chunk, with Lam_t the inclusive prefix sum of log alpha over
// tokens (per channel; Lam_{-1} = 0), Lp_t = Lam_{t-1}, L = Lam_63:
//   Lc[t][s] = [s < t] beta_s sum_i k_ti k_si exp(Lp_t,i - Lp_s,i)
//   Le[t][s] = [s < t] beta_s sum_i k_ti k_si exp(Lp_t,i - Lam_s,i)
//   P        = (beta o Ct)^T (I + Lc)^-1,   Ct[s][i] = k_si exp(L_i - Lp_s,i)
//   T_c      = diag(exp(L)) - P Ka,          Ka[t][j] = k_tj exp(Lp_t,j)
//   S_c      = Q V,  Q = (beta o Et)^T - P Le,  Et[s][i] = k_si exp(L_i - Lam_s,i)
// The Gram terms factor through a reference r = Lam_31 of the chunk,
// exp(Lp_t - Lp_s) = exp(Lp_t - r) exp(r - Lp_s), so that Lc and Le are one
// tensor-core product [Ck'; Ek'] Aq^T (Aq_t = k_t exp(Lp_t - r), Ck'_s = beta_s k_s
// exp(r - Lp_s), Ek'_s = beta_s k_s exp(r - Lam_s)); every factor stays finite while
// |Lam| <= 60 nats (times log2 e in the base-2 units used here).  A chunk beyond that
// (a channel decaying by more than e^60 within 64 tokens) is marked and its pair is
// formed token by token by the fp32 kernel instead.
//
// Products on tcgen05 with fp32 accumulation, every non-exact operand split into
// bf16 hi + lo (three products, lo ones first; V is exact bf16: two):
//   Gram^T [Ck'; Ek'] Aq^T (M = 128, N = 64, K = 128),  P (128 x 64, K = 64),
//   P Ka (128 x 128) and P Le (128 x 64) (K = 64),  Q V (128 x 128, K = 64).
// (I + Lc)^-1 is the blocked triangular inverse on CUDA cores.  Lanes of every
// accumulator are key channels i (or tokens s for the Gram), so each thread of the
// epilogue owns one row of T_c and S_c.
#include "dense_common.cuh"
#include "internal.cuh"
#include "sm100.cuh"

namespace hypic {
namespace {

using namespace sm100;
using dense::kLd;
using dense::split_pair;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kBox = kC * 128;                 // 64 channels x 64 tokens, bf16: 8 KB
constexpr int kThreads = 512;
constexpr int kCG = kThreads / 128;            // warps per TMEM lane quarter (column groups)
constexpr int kW64 = 64 / kCG;                 // columns of a 64-column accumulator per warp
constexpr int kW128 = 128 / kCG;
constexpr int kParts = kThreads / 128;         // token parts of the per-channel prefix
static_assert(kW64 == 16 || kW64 == 32, "a warp reads 16 or 32 columns of a 64-column accumulator");
constexpr float kMaxLog2 = 60.f * 1.4426950408889634f;   // |Lam| bound, base 2

// shared memory, from the 1024-aligned base
constexpr int kK = 0;                          // keys (token rows, two 64-channel boxes, 128-byte swizzle);
                                               // after the Gram: Le^T (rows s, t along K) hi, lo +8 KB
constexpr int kV = 2 * kBox;                   // values, the same layout
constexpr int kG = 4 * kBox;                   // the Gram operands, kept until Q is built:
constexpr int kGa = kG;                        //   [Ck'; Ek'] hi: channel half b is the 128-row tile at
                                               //   kGa + 16384 b (rows 0..63 Ck', 64..127 Ek'); lo +32 KB
constexpr int kGb = kG + 65536;                //   Aq hi (two boxes), lo +16 KB
constexpr int kX = kG + 98304;                 // the gates alpha (fp32 [64][128], TMA); then fp32 Lc, A =
                                               // (I + Lc)^-1 and temporaries; then P hi, lo +16 KB
constexpr int kLw = kX;
constexpr int kAw = kLw + kC * kLd * 4;
constexpr int kTw = kAw + kC * kLd * 4;
constexpr int kLam = kX + 32768;               // Lam, base 2, fp32 [65][128] (row 0 zero, row t + 1 = Lam_t)
                                               // while the Gram operands are built; then A's tiles, then Q
constexpr int kAi = kLam + 6144;               //   A (rows s, t along N) hi, lo +8 KB
constexpr int kQ = kLam;                       //   Q (rows i, s along K) hi, lo +16 KB
constexpr int kCtl = kLam + (kC + 1) * kD * 4;
constexpr int kStM = kG;                       // M_c staged for the TMA store: four 16 KB boxes of 32 columns
// S_c staged likewise, boxes 0, 1 over Aq's tiles and 2, 3 over Q's (the next chunk's
// gates arrive in kX meanwhile)
__host__ __device__ constexpr int st_s_box(int b) { return b < 2 ? kGb + 16384 * b : kQ + 16384 * (b - 2); }

struct Ctl {
    uint64_t full, mma, tdone, drain;
    float beta[kC];
    float eLr[kD];     // exp(L - r) per channel
    float er[kD];      // exp(r)
    float eL[kD];      // exp(L)
    float red[kThreads / 32];
    uint32_t tmem;
};
constexpr int kSmem = kCtl + (int)sizeof(Ctl) + 1024;
static_assert(kSmem <= 232448, "fits in one SM's shared memory");
static_assert(kTw + 3 * 256 * 4 <= kAi, "the inverse's temporaries end before A's tiles");
static_assert(kAi + 16384 <= kCtl && kQ + 32768 <= kCtl && kGb + 32768 <= kX, "tiles inside their regions");
static_assert(kAi % 1024 == 0 && kQ % 1024 == 0 && kX % 1024 == 0 && kGb % 1024 == 0, "tiles 1024-byte aligned");

// TMEM columns (256 allocated)
constexpr uint32_t kTG = 0;     // Gram^T (lanes s / 64 + s), then P Le (64), then Q V (128)
constexpr uint32_t kTP = 64;    // Ck'^T A (P before its row scale)
constexpr uint32_t kTT = 128;   // P Aq (P Ka before its column scale)

// byte offset of the 16-byte chunk c of row r in a 128-byte-swizzled tile
__device__ __forceinline__ int swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 8 fp32 values -> bf16 hi / lo 16-byte chunks at dst (lo at dst + lo_off)
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

// 4 values of row r, columns 4 c4 .. 4 c4 + 3 of a staged 128 x 128 fp32 result:
// box c4 / 8 (32 columns), chunk c4 % 8 of the 128-byte-swizzled row
__device__ __forceinline__ int st_m_box(int b) { return kStM + 16384 * b; }
template <bool S> __device__ __forceinline__ void stage4(uint8_t *smem, int r, int c4, float4 v) {
    const int b = c4 >> 3;
    *reinterpret_cast<float4 *>(smem + (S ? st_s_box(b) : st_m_box(b)) + swz(r, c4 & 7)) = v;
}

// W (16 or 32) consecutive columns of the warp's 32 lanes
template <int W> __device__ __forceinline__ void tmem_ldw(uint32_t taddr, uint32_t (&r)[W]) {
    if constexpr (W == 32) tmem_ld32(taddr, r);
    else tmem_ld16(taddr, r);
}

// One elected thread: three split products D (+)= A B over nk k-steps of 16,
// lo ones first (A_lo B_hi, A_hi B_lo, A_hi B_hi).
template <typename DescA, typename DescB>
__device__ __forceinline__ void mma3(uint32_t d, uint32_t idesc, int nk, DescA da, DescB db) {
    const int order[3][2] = {{1, 0}, {0, 1}, {0, 0}};
#pragma unroll
    for (int p = 0; p < 3; ++p)
        for (int ks = 0; ks < nk; ++ks)
            mma_f16(d, da(order[p][0], ks), db(order[p][1], ks), idesc, (p > 0 || ks > 0) ? 1u : 0u);
}

// One chunk of the launch: its pool row u (= work index), first token and length.
struct Item {
    int64_t u, c0;
    int l, h, nval;
};

// Work index w -> the chunk in slot w / H of its layer (false: no chunk uses the slot).
// Slot of chunk j of segment s: s + floor(t0_s / 64) + j.
__device__ __forceinline__ bool decode_item(const ScanArgs &a, int64_t slots, int64_t w, Item &it) {
    const int64_t per_layer = slots * a.H;
    const int l = (int)(w / per_layer);
    const int64_t rem = w % per_layer;
    const int64_t slot = rem / a.H;
    int lo = 0, hi = a.n_seg - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)mid + a.seg_offsets[mid] / kC <= slot) lo = mid;
        else hi = mid - 1;
    }
    const int64_t t0 = a.seg_offsets[lo], t1 = a.seg_offsets[lo + 1];
    const int64_t j = slot - (lo + t0 / kC);
    if (!(t0 >= 0 && t0 <= t1 && t1 <= a.N) || j < 0 || j * kC >= t1 - t0) return false;
    it.u = w;
    it.l = l;
    it.h = (int)(rem % a.H);
    it.c0 = t0 + j * kC;
    it.nval = (int)min((int64_t)kC, t1 - it.c0);
    return true;
}

// Persistent: each CTA walks the chunks w = blockIdx.x, + gridDim.x, ...  While a
// chunk's products and epilogues run, the next chunk's keys, gates and values are
// loaded into the regions that fall free (keys after P Le, gates after P Aq, values
// after Q V).
__global__ void __launch_bounds__(kThreads, 1)
    scan_kda_chunk_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_m,
                          const __grid_constant__ CUtensorMap tm_s, const ScanArgs a, int64_t slots,
                          float *pool_lam, int *steep_list) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align1024(smem_raw);
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + kCtl);
    float *lam = reinterpret_cast<float *>(smem + kLam);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n_items = (int64_t)a.n_layers * slots * a.H;

    // the next chunk at or after w in this CTA's stride
    auto find = [&](int64_t &w, Item &it) -> bool {
        for (; w < n_items; w += gridDim.x)
            if (decode_item(a, slots, w, it)) return true;
        return false;
    };
    auto row_of = [&](const Item &it) { return (int)((int64_t)it.l * a.N + it.c0); };
    auto beta_of = [&](const Item &it, int t) {
        return t < it.nval ? (a.beta ? a.beta[((int64_t)it.l * a.N + it.c0 + t) * a.H + it.h] : 1.f) : 0.f;
    };
    // (thread 0) the tiles of chunk it: keys, gates, values
    auto load_k = [&](const Item &it) {
        mbar_expect_tx(&ctl->full, (uint32_t)(4 * kBox + kC * kD * 4));
        tma_load_3d(smem + kK, &tm_k, &ctl->full, 0, it.h, row_of(it));
        tma_load_3d(smem + kK + kBox, &tm_k, &ctl->full, 64, it.h, row_of(it));
    };
    auto load_a = [&](const Item &it) { tma_load_3d(smem + kX, &tm_a, &ctl->full, 0, it.h, row_of(it)); };
    auto load_v = [&](const Item &it) {
        tma_load_3d(smem + kV, &tm_v, &ctl->full, 0, it.h, row_of(it));
        tma_load_3d(smem + kV + kBox, &tm_v, &ctl->full, 64, it.h, row_of(it));
    };

    int64_t w = blockIdx.x;
    Item cur;
    bool have = find(w, cur);
    if (tid == 0) {
        mbar_init(&ctl->full, 1);
        mbar_init(&ctl->mma, 1);
        mbar_init(&ctl->tdone, 1);
        mbar_init(&ctl->drain, 1);
        mbar_fence_init();
        if (have) {
            load_k(cur);
            load_a(cur);
            load_v(cur);
        }
    }
    if (warp == 0) tmem_alloc(&ctl->tmem, 256);
    if (have && tid >= kD && tid < kD + kC) ctl->beta[tid - kD] = beta_of(cur, tid - kD);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    const int q4 = warp & 3, cg = warp >> 2;         // TMEM lane quarter, column group
    const int m = q4 * 32 + lane;                    // accumulator row of this thread
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    float *Lw = reinterpret_cast<float *>(smem + kLw);
    float *Aw = reinterpret_cast<float *>(smem + kAw);
    float *Tw = reinterpret_cast<float *>(smem + kTw);
    const float ln2 = 0.6931471805599453f;
    uint32_t full_par = 0, t_par = 0, mma_phase = 0;
    bool ok = true, pending = have;   // pending: loads in flight on `full`

    while (have && ok) {
        int64_t wn = w + gridDim.x;
        Item nxt;
        const bool have_n = find(wn, nxt);
        float bnext = 0.f;   // the next chunk's beta (threads kD .. kD + 63)
        // the previous chunk's TMA stores have read their staging tiles (Gram, Q and Lam regions)
        if (tid == 0) bulk_wait_read_all();
        ok = __syncthreads_and(mbar_wait(&ctl->full, full_par));   // this chunk's tiles
        full_par ^= 1u;
        pending = false;
        if (!ok) break;
        const int64_t u = cur.u;
        const int nval = cur.nval;

        // ---- gates: Lam (base 2), the prefix over tokens per channel; tokens past the
        // segment's end get alpha = 1 and beta = 0 (their keys then act on nothing)
        float mx = 0.f;
        {
            const float4 *a4 = reinterpret_cast<const float4 *>(smem + kX);
            float4 *g4 = reinterpret_cast<float4 *>(lam + kD);
#pragma unroll
            for (int i = 0; i < kC * kD / 4 / kThreads; ++i) {
                const int f = tid + kThreads * i;   // float4 index: token f / 32
                const bool v = (f >> 5) < nval;
                const float4 x = a4[f];
                g4[f] = v ? make_float4(log2f(x.x), log2f(x.y), log2f(x.z), log2f(x.w)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (tid < kD) lam[tid] = 0.f;
            __syncthreads();
            constexpr int kTok = kC / kParts;                  // tokens of a part
            const int ch = tid & (kD - 1), part = tid >> 7;   // tokens kTok part .. kTok part + kTok - 1
            float acc = 0.f;
#pragma unroll 8
            for (int t = part * kTok; t < part * kTok + kTok; ++t) {
                acc += lam[(t + 1) * kD + ch];
                lam[(t + 1) * kD + ch] = acc;
            }
            __syncthreads();
            float base = 0.f;   // the totals of the earlier parts
            for (int q = 0; q < part; ++q) base += lam[(q + 1) * kTok * kD + ch];
            __syncthreads();
#pragma unroll 8
            for (int t = part * kTok; t < part * kTok + kTok; ++t) {
                const float x = lam[(t + 1) * kD + ch] + base;
                if (part) lam[(t + 1) * kD + ch] = x;
                mx = fmaxf(mx, fabsf(x));
            }
            if (!(mx <= kMaxLog2)) mx = INFINITY;   // a NaN gate counts as steep
        }
        const bool is_steep = __syncthreads_or(mx > kMaxLog2);
        if (is_steep) {   // listed: its pair comes from the token-by-token kernel; nothing here is in use
            if (tid == 0) steep_list[1 + atomicAdd(steep_list, 1)] = (int)u;
            if (have_n) {
                if (tid == 0) {
                    load_k(nxt);
                    load_a(nxt);
                    load_v(nxt);
                }
                pending = true;
                if (tid >= kD && tid < kD + kC) ctl->beta[tid - kD] = beta_of(nxt, tid - kD);
            }
            __syncthreads();
            w = wn;
            cur = nxt;
            have = have_n;
            continue;
        }
        if (tid < kD) {   // per-channel factors of the scales below (r = Lam_31, L = Lam_63)
            const float r = lam[32 * kD + tid], L = lam[kC * kD + tid];
            ctl->eLr[tid] = exp2f(L - r);
            ctl->er[tid] = exp2f(r);
            ctl->eL[tid] = exp2f(L);
        }

        // ---- the Gram operands (bf16 hi / lo, 128-byte swizzle): Aq_t = k_t e^(Lp_t - r),
        // Ck'_s = beta_s k_s e^(r - Lp_s), Ek'_s = beta_s k_s e^(r - Lam_s).  They are kept:
        // beta o Ct = Ck' diag(e^(L - r)), Ka = Aq diag(e^r), beta o Et = Ek' diag(e^(L - r)).
        const uint8_t *kt = smem + kK;
#pragma unroll 1
        for (int f = tid; f < kC * 16; f += kThreads) {
            const int t = f >> 4, cc = f & 15, b = cc >> 3, c = cc & 7, chn = cc * 8;
            const uint4 raw = *reinterpret_cast<const uint4 *>(kt + b * kBox + swz(t, c));
            const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
            float lp[8], lt[8], rf[8];
            load8(lam + t * kD + chn, lp);
            load8(lam + (t + 1) * kD + chn, lt);
            load8(lam + 32 * kD + chn, rf);
            const float bt = ctl->beta[t];
            float aq[8], ck[8], ek[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float kv = (e & 1) ? bf_hi(wv[e >> 1]) : bf_lo(wv[e >> 1]);
                aq[e] = kv * exp2f(lp[e] - rf[e]);
                ck[e] = bt * kv * exp2f(rf[e] - lp[e]);
                ek[e] = bt * kv * exp2f(rf[e] - lt[e]);
            }
            put8(smem + kGb + b * kBox + swz(t, c), 16384, aq);
            put8(smem + kGa + b * 16384 + swz(t, c), 32768, ck);
            put8(smem + kGa + b * 16384 + swz(kC + t, c), 32768, ek);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {   // Gram^T = [Ck'; Ek'] Aq^T (M = 128, N = 64, K = 128)
            tc_fence_after();
            constexpr uint32_t id_g = idesc_bf16_f32(128, 64, false, false);
            const uint32_t ga = smem_addr(smem + kGa), gb = smem_addr(smem + kGb);
            const uint64_t dga = smem_desc_sw128(ga, 0, 1024), dgb = smem_desc_sw128(gb, 0, 1024);
            mma3(tmem + kTG, id_g, 8,
                 [&](int hl, int ks) {
                     return dga + (uint64_t)(hl * 2048 + (ks >> 2) * 1024 + (ks & 3) * 2);
                 },
                 [&](int hl, int ks) {
                     return dgb + (uint64_t)(hl * 1024 + (ks >> 2) * (kBox >> 4) + (ks & 3) * 2);
                 });
            mma_commit(&ctl->mma);
        }
        ok = __syncthreads_and(mbar_wait(&ctl->mma, mma_phase));
        mma_phase ^= 1u;
        tc_fence_after();
        if (!ok) break;

        {   // ---- Lc (fp32, for the inverse) and Le^T (bf16 hi / lo, over the keys), t > s only
            uint32_t r[kW64];
            tmem_ldw<kW64>(tmem + lane_off + kTG + (uint32_t)(cg * kW64), r);
            tmem_wait_ld();
            if (q4 < 2) {
                const int s = m;
#pragma unroll
                for (int i = 0; i < kW64; ++i) {
                    const int t = cg * kW64 + i;
                    Lw[t * kLd + s] = t > s ? __uint_as_float(r[i]) : 0.f;
                }
            } else {
                const int s = m - kC;
#pragma unroll
                for (int cc = 0; cc < kW64 / 8; ++cc) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int t = cg * kW64 + cc * 8 + e;
                        x[e] = t > s ? __uint_as_float(r[cc * 8 + e]) : 0.f;
                    }
                    put8(smem + kK + swz(s, cg * (kW64 / 8) + cc), 8192, x);
                }
            }
        }
        __syncthreads();
        dense::tri_inverse<kThreads, 1, true, true>(Lw, Aw, Tw, tid);
        // ---- A -> bf16 hi / lo (rows s, t contiguous: the MN-major B of Ck'^T A)
#pragma unroll
        for (int i = 0; i < kC * 8 / kThreads; ++i) {
            const int f = tid + kThreads * i;
            const int s = f >> 3, c = f & 7;
            float x[8];
            load8(Aw + s * kLd + c * 8, x);
            put8(smem + kAi + swz(s, c), 8192, x);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {   // Ck'^T A (M = 128 channels, N = 64, K = 64): Ck' read MN-major from the Gram tile
            tc_fence_after();
            constexpr uint32_t id_p = idesc_bf16_f32(128, 64, true, true);
            const uint32_t ga = smem_addr(smem + kGa), ab = smem_addr(smem + kAi);
            const uint64_t dga = smem_desc_sw128(ga, 16384, 1024), dab = smem_desc_sw128(ab, 8192, 1024);
            mma3(tmem + kTP, id_p, 4,
                 [&](int hl, int ks) { return dga + (uint64_t)(hl * 2048 + ks * 128); },
                 [&](int hl, int ks) { return dab + (uint64_t)(hl * 512 + ks * 128); });
            mma_commit(&ctl->mma);
        }
        ok = __syncthreads_and(mbar_wait(&ctl->mma, mma_phase));
        mma_phase ^= 1u;
        tc_fence_after();
        if (!ok) break;

        {   // ---- P = diag(e^(L - r)) Ck'^T A -> bf16 hi / lo (rows i, t along K)
            uint32_t r[kW64];
            tmem_ldw<kW64>(tmem + lane_off + kTP + (uint32_t)(cg * kW64), r);
            const float sc = ctl->eLr[m];
            tmem_wait_ld();
#pragma unroll
            for (int cc = 0; cc < kW64 / 8; ++cc) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = sc * __uint_as_float(r[cc * 8 + e]);
                put8(smem + kX + swz(m, cg * (kW64 / 8) + cc), 16384, x);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {   // P Le first (Q waits on it), then P Aq (the epilogue of T_c)
            tc_fence_after();
            constexpr uint32_t id_t = idesc_bf16_f32(128, 128, false, true);
            constexpr uint32_t id_l = idesc_bf16_f32(128, 64, false, false);
            const uint32_t pb = smem_addr(smem + kX), gb = smem_addr(smem + kGb), lb = smem_addr(smem + kK);
            const uint64_t dpb = smem_desc_sw128(pb, 0, 1024), dlb = smem_desc_sw128(lb, 0, 1024),
                           dgb = smem_desc_sw128(gb, kBox, 1024);
            auto pd = [&](int hl, int ks) { return dpb + (uint64_t)(hl * 1024 + ks * 2); };
            mma3(tmem + kTG, id_l, 4, pd, [&](int hl, int ks) { return dlb + (uint64_t)(hl * 512 + ks * 2); });
            mma_commit(&ctl->mma);
            mma3(tmem + kTT, id_t, 4, pd, [&](int hl, int ks) { return dgb + (uint64_t)(hl * 1024 + ks * 128); });
            mma_commit(&ctl->tdone);
        }
        ok = __syncthreads_and(mbar_wait(&ctl->mma, mma_phase));
        mma_phase ^= 1u;
        tc_fence_after();
        if (!ok) break;
        // the keys' region (Le^T) is free: the next chunk's keys; its beta in flight too
        if (have_n) {
            if (tid == 0) load_k(nxt);
            pending = true;
            if (tid >= kD && tid < kD + kC) bnext = beta_of(nxt, tid - kD);
        }

        const int i = m;
        uint32_t r[32];
        {   // ---- Q[i][s] = e^(L_i - r_i) Ek'[s][i] - (P Le)[i][s] -> bf16 hi / lo (rows i, s along K)
            tmem_ldw<kW64>(tmem + lane_off + kTG + (uint32_t)(cg * kW64), *reinterpret_cast<uint32_t(*)[kW64]>(r));
            const float sc = ctl->eLr[i];
            const uint8_t *ecol = smem + kGa + (i >> 6) * 16384 + ((i & 7) << 1);   // Ek' rows 64 + s
            const int ci = (i & 63) >> 3;
            tmem_wait_ld();
#pragma unroll
            for (int cc = 0; cc < kW64 / 8; ++cc) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int s = cg * kW64 + cc * 8 + e;
                    const int off = swz(kC + s, ci);
                    const float ek =
                        __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t *>(ecol + off) << 16) +
                        __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t *>(ecol + 32768 + off) << 16);
                    x[e] = sc * ek - __uint_as_float(r[cc * 8 + e]);
                }
                put8(smem + kQ + swz(i, cg * (kW64 / 8) + cc), 16384, x);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {   // S_c = Q V (V exact in bf16: Q_lo V, then Q_hi V)
            tc_fence_after();
            constexpr uint32_t id_z = idesc_bf16_f32(128, 128, false, true);
            const uint32_t qb = smem_addr(smem + kQ), vb = smem_addr(smem + kV);
            const uint64_t dqb = smem_desc_sw128(qb, 0, 1024), dvb = smem_desc_sw128(vb, kBox, 1024);
#pragma unroll
            for (int hl = 1; hl >= 0; --hl)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16(tmem + kTG, dqb + (uint64_t)(hl * 1024 + ks * 2), dvb + (uint64_t)(ks * 128), id_z,
                            (hl == 0 || ks > 0) ? 1u : 0u);
            mma_commit(&ctl->mma);
        }
        // ---- T_c = diag(e^L) - (P Aq) diag(e^r), scaled by a power of two to max |M_c| in [1, 2)
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl->tdone, t_par));   // warp-uniform: TMEM loads are collective
        t_par ^= 1u;
        tc_fence_after();
        if (ok && have_n && tid == 0) load_a(nxt);   // P's tiles are read: the next chunk's gates
        float tmx = 0.f;
        const float di = ctl->eL[i];
        if (ok) {
#pragma unroll
            for (int p = 0; p < kW128 / 32; ++p) {
                tmem_ld32(tmem + lane_off + kTT + (uint32_t)(cg * kW128 + p * 32), r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int col = cg * kW128 + p * 32 + e;
                    tmx = fmaxf(tmx, fabsf((col == i ? di : 0.f) - ctl->er[col] * __uint_as_float(r[e])));
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) tmx = fmaxf(tmx, __shfl_xor_sync(0xffffffffu, tmx, off));
        if (lane == 0) ctl->red[warp] = tmx;
        ok = __syncthreads_and(ok);
        if (!ok) break;
        {
            tmx = 0.f;
#pragma unroll
            for (int wi = 0; wi < kThreads / 32; ++wi) tmx = fmaxf(tmx, ctl->red[wi]);
            const int ex = dense::exponent_of(tmx);
            const float scl = ldexpf(1.f, -ex);
#pragma unroll
            for (int p = 0; p < kW128 / 32; ++p) {
                tmem_ld32(tmem + lane_off + kTT + (uint32_t)(cg * kW128 + p * 32), r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    float4 v;
                    float *vp = &v.x;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int col = cg * kW128 + p * 32 + e + q;
                        vp[q] = ((col == i ? di : 0.f) - ctl->er[col] * __uint_as_float(r[e + q])) * scl;
                    }
                    stage4<false>(smem, i, (cg * kW128 + p * 32 + e) >> 2, v);
                }
            }
            fence_async_smem();
            __syncthreads();
            if (tid == 0) {
#pragma unroll
                for (int b = 0; b < 4; ++b) tma_store_3d(&tm_m, smem + st_m_box(b), 32 * b, 0, (int)(u * kD));
                bulk_commit();
                pool_lam[u] = (float)ex * ln2;
            }
        }
        ok = __syncthreads_and(mbar_wait(&ctl->mma, mma_phase));   // S_c is done
        mma_phase ^= 1u;
        tc_fence_after();
        if (!ok) break;
        if (have_n && tid == 0) load_v(nxt);   // the values are read: the next chunk's
        // ---- S_c
#pragma unroll
        for (int p = 0; p < kW128 / 32; ++p) {
            tmem_ld32(tmem + lane_off + kTG + (uint32_t)(cg * kW128 + p * 32), r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; e += 4)
                stage4<true>(smem, m, (cg * kW128 + p * 32 + e) >> 2,
                       make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                                   __uint_as_float(r[e + 3])));
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int b = 0; b < 4; ++b) tma_store_3d(&tm_s, smem + st_s_box(b), 32 * b, 0, (int)(u * kD));
            bulk_commit();
        }
        if (have_n && tid >= kD && tid < kD + kC) ctl->beta[tid - kD] = bnext;   // this chunk's beta is done
        w = wn;
        cur = nxt;
        have = have_n;
    }

    if (!ok && tid == 0) {   // a wait gave up: drain this thread's MMAs and loads, then report
        mma_commit(&ctl->drain);
        mbar_wait(&ctl->drain, 0);
        if (pending) mbar_wait(&ctl->full, full_par);
        if (a.d_err) atomicExch(a.d_err, (int)HYPIC_ETIMEOUT);
    }
    if (tid == 0) bulk_wait_all();   // the staged tiles are read and the stores complete
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// Per (layer, segment): the first pool row of its chunks and their count; per chunk
// slot p (and p = slots): the first token of the chunk in that slot, or for a slot no
// chunk uses, the end of the segment before it -- monotone, so that the chunks form
// a segment list for the token-by-token kernel.
__global__ void kda_index_kernel(const ScanArgs a, int64_t slots, int32_t *seg_first, int32_t *chain_len,
                                 int64_t *voffs, int *steep_list) {
    const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x == 0) *steep_list = 0;   // the count of chunks listed for the token-by-token kernel
    const int64_t R = (int64_t)a.n_layers * a.n_seg;
    if (x < R) {
        const int l = (int)(x / a.n_seg), seg = (int)(x % a.n_seg);
        int64_t t0 = a.seg_offsets[seg], t1 = a.seg_offsets[seg + 1];
        if (!(t0 >= 0 && t0 <= t1 && t1 <= a.N)) {
            if (l == 0) flag_index_error(a.d_err);
            t0 = t1 = 0;
        }
        seg_first[x] = (int32_t)((int64_t)l * slots + seg + t0 / kC);
        chain_len[x] = (int32_t)((t1 - t0 + kC - 1) / kC);
    }
    if (x <= slots) {
        int lo = 0, hi = a.n_seg - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)mid + a.seg_offsets[mid] / kC <= x) lo = mid;
            else hi = mid - 1;
        }
        const int64_t t0 = a.seg_offsets[lo], t1 = a.seg_offsets[lo + 1];
        const int64_t j = x - (lo + t0 / kC);
        voffs[x] = j < 0 ? t0 : (j * kC < t1 - t0 ? t0 + j * kC : t1);
    }
}

struct KdaLayout {
    int64_t slots, P;
    int64_t M, S, lam, steep, voffs, first, len, total;   // byte offsets
};

int64_t up256(int64_t b) { return (b + 255) / 256 * 256; }

KdaLayout kda_layout(const ScanArgs &a) {
    KdaLayout t{};
    t.slots = (int64_t)a.n_seg + a.N / kC;
    t.P = (int64_t)a.n_layers * t.slots;
    const int64_t rows = t.P * a.H;
    const int64_t R = (int64_t)a.n_layers * a.n_seg;
    int64_t o = 0;
    t.M = o;      o += up256(rows * kD * kD * 4);
    t.S = o;      o += up256(rows * kD * kD * 4);
    t.lam = o;    o += up256(rows * 4);
    t.steep = o;  o += up256((rows + 1) * 4);   // count, then the listed pool rows
    t.voffs = o;  o += up256((t.slots + 1) * 8);
    t.first = o;  o += up256(R * 4);
    t.len = o;    o += up256(R * 4);
    t.total = o;
    return t;
}

}  // namespace

bool scan_kda_tc_shape(const ScanArgs &a) {
    if (!(a.fam == HYPIC_KDA && a.in_dtype == HYPIC_BF16 && a.dk == kD && a.dv == kD && a.o_out == nullptr &&
          a.N > 0 && a.n_layers > 0 && a.n_seg > 0 && a.n_layers <= 65535))
        return false;
    const int64_t slots = (int64_t)a.n_seg + a.N / kC;
    const int64_t rows = (int64_t)a.n_layers * slots * a.H;
    return (int64_t)a.n_layers * a.N < ((int64_t)1 << 31) && slots * a.H < ((int64_t)1 << 31) &&
           rows * kD < ((int64_t)1 << 31) && (int64_t)a.n_layers * a.n_seg * a.H < ((int64_t)1 << 30) &&
           kda_layout(a).total <= kKdaMaxScratch;
}

bool scan_kda_tc_supported(const ScanArgs &a) { return scan_kda_tc_shape(a) && tensor_map_encoder() != nullptr; }

int64_t scan_kda_tc_bytes(const ScanArgs &a) { return kda_layout(a).total; }

cudaError_t launch_scan_kda_tc(const ScanArgs &a, cudaStream_t s) {
    const KdaLayout t = kda_layout(a);
    uint8_t *ws = reinterpret_cast<uint8_t *>(a.ws);
    float *pM = reinterpret_cast<float *>(ws + t.M), *pS = reinterpret_cast<float *>(ws + t.S);
    float *plam = reinterpret_cast<float *>(ws + t.lam);
    int *steep = reinterpret_cast<int *>(ws + t.steep);   // [0]: count, then pool rows
    int64_t *voffs = reinterpret_cast<int64_t *>(ws + t.voffs);
    int32_t *first = reinterpret_cast<int32_t *>(ws + t.first), *clen = reinterpret_cast<int32_t *>(ws + t.len);
    const int64_t R = (int64_t)a.n_layers * a.n_seg;

    const int64_t nidx = R > t.slots + 1 ? R : t.slots + 1;
    kda_index_kernel<<<(unsigned)((nidx + 255) / 256), 256, 0, s>>>(a, t.slots, first, clen, voffs, steep);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    const uint64_t rows = (uint64_t)a.n_layers * (uint64_t)a.N;
    const uint64_t prow = (uint64_t)t.P * a.H * kD;   // pool rows of 128 floats
    CUtensorMap mk, mv, ma, mm, ms;
    if (!make_tensor_map_3d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k, kD, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v, kD, a.H, rows, 64, kC,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.alpha, kD, a.H, rows, kD, kC,
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tensor_map_3d(&mm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, pM, kD, 1, prow, 32, kD,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, pS, kD, 1, prow, 32, kD,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(scan_kda_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = 148;
    const int64_t items = t.P * a.H;   // one CTA per SM walks the chunks
    const unsigned grid = (unsigned)(items < sms ? items : sms);
    scan_kda_chunk_kernel<<<grid, kThreads, kSmem, s>>>(mk, mv, ma, mm, ms, a, t.slots, plam, steep);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // chunks too steep for the factored Gram (listed by the chunk kernel): their pairs
    // token by token, a few CTAs walking the list
    ScanArgs f = a;
    f.n_seg = (int)t.slots;
    f.seg_offsets = voffs;
    f.lam_out = plam;
    f.M_out = pM;
    f.S_out = pS;
    f.ws = nullptr;
    f.unit_list = steep + 1;
    f.unit_count = steep;
    e = launch_scan_recurrent(f, s);
    if (e != cudaSuccess) return e;

    // each segment: its chunks' pairs in order
    ChainArgs c{};
    c.fam = HYPIC_DENSE;   // (lambda, M) pairs
    c.R = (int)R;
    c.n_layers = 1;
    c.H = a.H;
    c.dk = kD;
    c.dv = kD;
    c.max_chain = (int)((a.N + kC - 1) / kC);
    c.P = (int)t.P;
    c.chain_len = clen;
    c.seg_idx = nullptr;
    c.seg_first = first;
    c.pool_lam = plam;
    c.pool_M = pM;
    c.pool_S = pS;
    c.S_init = nullptr;
    c.S_out = a.S_out;
    c.d_err = a.d_err;
    c.two_way = 1;   // the chunk pairs carry ~1e-5 from bf16 inputs; two-way splits keep the chains at ~1e-5
    return launch_compose_prefix(c, a.lam_out, a.M_out, s);
}

}  // namespace hypic
