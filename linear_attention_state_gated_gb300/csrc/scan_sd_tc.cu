// scan_sd_tc.cu -- scalar / diagonal segment scan on tcgen05 tensor cores.
//
// For a diagonal (or scalar) transition the zero-start final state of a
// segment of L tokens is
//     S(C|0) = sum_s w_s (beta_s k_s) v_s^T,   w_{s,i} = prod_{r > s} alpha_{r,i},
// i.e. a plain sum of rank-1 terms whose weights are the products of the
// gates of all LATER tokens.  Walking the segment's chunks from the end
// backwards, the running product over later tokens is known when a chunk is
// processed, so every chunk adds  K~^T V  (K~ = weighted keys) into the same
// fp32 TMEM accumulator with no rescaling of the accumulator at all; the
// transition is lambda = sum_t log alpha_t (log alpha per channel for diag).
//
// Per CTA one (layer, segment, head) chain -- or, with scratch, an equal share
// of all chains' chunks (see the work pieces below) -- d_k = d_v = 128:
//   warp 0       TMA producer: K, V (and the diagonal gates) of a chunk of C
//                tokens into a ring of NS shared-memory stages (128B swizzle);
//   warps 2..    TW "weighting" warps: K~ = w * beta * k, split exactly into
//                bf16 hi + lo (K~ - hi), hi written over K, lo into a separate
//                tile, same swizzled positions; at the end the epilogue
//                (TMEM -> S rows);
//   warp 1       one thread issues tcgen05.mma: D[128x128] += K~hi^T V + K~lo^T V
//                (both operands MN-major, M = key channel, N = value channel,
//                K = token) and commits each stage back to the producer.
// V is used exactly (bf16 input); the hi/lo split keeps K~ to ~2^-17 relative.
// Scalar gates: per-token log alpha, suffix sums by warp shuffles, Kahan-summed
// lambda.  Diagonal gates: per channel, the running product of later gates
// (underflow to 0 is the right limit for a weight); lambda from the logs of
// products over groups of rows.  Every wait is time-bounded; a timeout is
// reported as HYPIC_ETIMEOUT.
#include "internal.cuh"
#include "sm100.cuh"

namespace hypic {
namespace {

using namespace sm100;

constexpr int kTmemCols = 128;

template <int FAM, int C, int NS, int TW>
struct SdCfg {
    static constexpr int THREADS = 64 + 32 * TW;
    static constexpr int WT = 32 * TW;                     // weighting threads
    static constexpr int BOX = C * 128;                    // 64 channels x C tokens, bf16
    static constexpr int TILE = 2 * BOX;                   // 128 channels
    static constexpr int ATILE = FAM == HYPIC_DIAG ? C * 512 : 0;   // fp32 gates
    static constexpr int STAGE = 2 * TILE + ATILE;         // TMA ring stage: K (-> K~hi), V, gates
    static constexpr uint32_t TX = STAGE;                  // bytes TMA brings per stage
    static constexpr int LO = NS * STAGE;                  // two K~lo tiles (chunk parity) after the ring
    static constexpr int NG = WT / 64;                     // diag: row groups (64 channel pairs each)
    static constexpr int RPG = C / NG;                     // diag: rows per group
    static_assert(C == 32 || C == 64, "chunk of 32 or 64 tokens");
    static_assert(NS >= 2 && NS <= 8, "2 to 8 stages");
    static_assert(TW == 4 || TW == 8, "4 or 8 weighting warps");
    static_assert(STAGE % 1024 == 0, "stages stay 1024-byte aligned");
    static_assert((16 * C) % WT == 0, "whole 16-byte chunks per thread");
};

constexpr int kMaxBalSeg = 512;   // segments the balanced schedule indexes in shared memory

struct SdCtrl {
    uint64_t full[8], ready[8], empty[8], lofree[2], accf, drain;
    float rowf[2][64];          // per-row factor of the chunk (weight * beta, or beta)
    float2 gprod[2][4][64];     // diag: gate product of each row group per channel pair
    float2 lamp[4][64];         // diag: per-group partial lambda
    int pre[kMaxBalSeg + 1];    // balanced schedule: chunks of the segments before s
    uint32_t tmem;
    int abort;
};

// ring + two lo tiles + control block + slack for the 1024-byte alignment
template <int FAM, int C, int NS, int TW>
constexpr int sd_smem_bytes() {
    using Cfg = SdCfg<FAM, C, NS, TW>;
    return Cfg::LO + 2 * Cfg::TILE + (int)sizeof(SdCtrl) + 1024;
}

__device__ __forceinline__ float warp_suffix_incl(float x, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, x, off);
        if (lane + off < 32) x += y;
    }
    return x;
}

__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t *>(&v); }

// Two fp32 values -> bf16 hi pair and bf16 lo pair (x = hi + lo to ~2^-17 relative).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
    const __nv_bfloat162 ll = __floats2bfloat162_rn(x0 - __low2float(hh), x1 - __high2float(hh));
    hi = bf2_bits(hh);
    lo = bf2_bits(ll);
}

__device__ __forceinline__ void split8(const uint4 raw, const float w, uint4 &hi, uint4 &lo) {
    const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t h[4], l[4];
#pragma unroll
    for (int p = 0; p < 4; ++p)
        split2(__uint_as_float(in[p] << 16) * w, __uint_as_float(in[p] & 0xFFFF0000u) * w, h[p], l[p]);
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void kahan(float &sum, float &comp, float v) {
    const float y = v - comp;
    const float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
}

// log of a product of gates; exact fallback when the product left the normal range
__device__ __forceinline__ float log_group(float prod, const float *a, int n, int stride) {
    if (prod >= 0x1p-100f) return logf(prod);
    float s = 0.f;
    for (int i = 0; i < n; ++i) s += logf(a[i * stride]);
    return s;
}

// ---------------------------------------------------------------- work pieces
// One chain (layer, segment, head) is split into chunks of C tokens numbered
// from the segment's END (chunk j covers tokens [t1 - (j+1) C, t1 - j C)).
// Unbalanced schedule: CTA u takes all chunks of chain u.  Balanced schedule:
// the chains' chunk lists are concatenated in (layer, segment, head) order and
// CTA g of G takes the positions [g N / G, (g+1) N / G); a piece is the part of
// one chain inside that range.  A piece that is a whole chain writes the
// chain's (lambda, S); the others write partial results to the scratch slot
// (g, 0) -- the piece starting at the range's first position -- or (g, 1), and
// sd_combine_kernel folds them.
struct Piece {
    int l, seg, h, nc, jb, je, slot;
    int64_t t0, t1;
    bool whole;
};

// scratch slot: lambda (128 floats) then S (128 x 128)
constexpr int kSlotFloats = 128 + 128 * 128;

__device__ __forceinline__ void seg_bounds(const ScanArgs &a, int seg, int64_t &t0, int64_t &t1, bool &bad) {
    t0 = a.seg_offsets[seg];
    t1 = a.seg_offsets[seg + 1];
    bad = !(t0 >= 0 && t0 <= t1 && t1 <= a.N);
    if (bad) t0 = t1 = 0;
}

// chunks per segment, prefix over segments, built by one warp
template <int C>
__device__ __forceinline__ void build_prefix(const ScanArgs &a, int *pre, int lane) {
    int carry = 0;
    for (int base = 0; base < a.n_seg; base += 32) {
        const int sg = base + lane;
        int v = 0;
        if (sg < a.n_seg) {
            int64_t t0, t1;
            bool bad;
            seg_bounds(a, sg, t0, t1, bad);
            v = (int)((t1 - t0 + C - 1) / C);
        }
        int x = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (sg < a.n_seg) pre[sg + 1] = carry + x;
        carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) pre[0] = 0;
}

// the piece that starts at concatenated position pos (b0 <= pos < b1)
template <int C>
__device__ __forceinline__ Piece piece_at(const ScanArgs &a, const int *pre, int64_t pos, int64_t b0, int64_t b1) {
    Piece p;
    const int NC = pre[a.n_seg];
    const int64_t per_layer = (int64_t)a.H * NC;
    p.l = (int)(pos / per_layer);
    const int64_t rem = pos - (int64_t)p.l * per_layer;
    int lo = 0, hi = a.n_seg - 1;   // last segment whose chunks start at or before rem
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)a.H * pre[mid] <= rem) lo = mid;
        else hi = mid - 1;
    }
    p.seg = lo;
    p.nc = pre[lo + 1] - pre[lo];
    const int64_t rem2 = rem - (int64_t)a.H * pre[lo];
    p.h = (int)(rem2 / p.nc);
    p.jb = (int)(rem2 % p.nc);
    const int64_t u0 = pos - p.jb;
    p.je = (int)(b1 - u0 < (int64_t)p.nc ? b1 - u0 : (int64_t)p.nc);
    p.whole = p.jb == 0 && p.je == p.nc;
    p.slot = pos == b0 ? 0 : 1;
    bool bad;
    seg_bounds(a, p.seg, p.t0, p.t1, bad);
    return p;
}

template <int FAM, int C, int NS, int TW, bool BAL>
__global__ void __launch_bounds__(SdCfg<FAM, C, NS, TW>::THREADS, 2)
    scan_sd_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_a, const ScanArgs a) {
    using Cfg = SdCfg<FAM, C, NS, TW>;
    constexpr bool kDiag = FAM == HYPIC_DIAG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align1024(smem_raw);
    SdCtrl *ctl = reinterpret_cast<SdCtrl *>(smem + Cfg::LO + 2 * Cfg::TILE);
    volatile int *abortp = &ctl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->ready[s], TW);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->lofree[0], 1);
        mbar_init(&ctl->lofree[1], 1);
        mbar_init(&ctl->accf, 1);
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        mbar_fence_init();
        tma_prefetch(&tm_k);
        tma_prefetch(&tm_v);
        if (kDiag) tma_prefetch(&tm_a);
    }
    if (BAL && warp == 0) build_prefix<C>(a, ctl->pre, lane);
    if (warp == 1) tmem_alloc(&ctl->tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;

    // this CTA's range of concatenated chunk positions
    int64_t b0, b1;
    if (BAL) {
        const int64_t total = (int64_t)a.n_layers * a.H * ctl->pre[a.n_seg];
        b0 = (int64_t)blockIdx.x * total / gridDim.x;
        b1 = ((int64_t)blockIdx.x + 1) * total / gridDim.x;
    } else {
        b0 = 0;
        b1 = 1;   // one piece: the whole chain of this CTA
    }
    auto piece = [&](int64_t pos) -> Piece {
        if (BAL) return piece_at<C>(a, ctl->pre, pos, b0, b1);
        Piece p;
        const int unit = blockIdx.x;
        p.h = unit % a.H;
        p.seg = (unit / a.H) % a.n_seg;
        p.l = unit / (a.H * a.n_seg);
        bool bad;
        seg_bounds(a, p.seg, p.t0, p.t1, bad);
        if (bad && threadIdx.x == 0) flag_index_error(a.d_err);
        p.nc = (int)((p.t1 - p.t0 + C - 1) / C);
        p.jb = 0;
        p.je = p.nc;
        p.whole = true;
        p.slot = 0;
        return p;
    };
    auto advance = [&](const Piece &p) -> int64_t { return BAL ? (int64_t)(p.je - p.jb) : 1; };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int c = 0;   // chunks of this CTA so far (ring position)
            for (int64_t pos = b0; pos < b1 && !*abortp;) {
                const Piece p = piece(pos);
                const int64_t row_end = (int64_t)p.l * a.N + p.t1;   // token row just past the segment
                for (int j = p.jb; j < p.je; ++j, ++c) {
                    const int s = c % NS;
                    const uint32_t ph = (uint32_t)(c / NS) & 1u;
                    if (!mbar_wait(&ctl->empty[s], ph ^ 1u) || *abortp) {
                        *abortp = 1;
                        break;
                    }
                    uint8_t *st = smem + s * Cfg::STAGE;
                    const int row = (int)(row_end - (int64_t)(j + 1) * C);
                    mbar_expect_tx(&ctl->full[s], Cfg::TX);
                    tma_load_3d(st, &tm_k, &ctl->full[s], 0, p.h, row);
                    tma_load_3d(st + Cfg::BOX, &tm_k, &ctl->full[s], 64, p.h, row);
                    tma_load_3d(st + Cfg::TILE, &tm_v, &ctl->full[s], 0, p.h, row);
                    tma_load_3d(st + Cfg::TILE + Cfg::BOX, &tm_v, &ctl->full[s], 64, p.h, row);
                    if (kDiag) tma_load_3d(st + 2 * Cfg::TILE, &tm_a, &ctl->full[s], 0, p.h, row);
                }
                pos += advance(p);
            }
            if (*abortp) {   // let copies already in flight land before the CTA leaves
                for (int cc = c - NS < 0 ? 0 : c - NS; cc < c; ++cc)
                    mbar_wait(&ctl->full[cc % NS], (uint32_t)(cc / NS) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 128, true, true);
            int c = 0;
            for (int64_t pos = b0; pos < b1 && !*abortp;) {
                const Piece p = piece(pos);
                for (int j = p.jb; j < p.je; ++j, ++c) {
                    const int s = c % NS;
                    const uint32_t ph = (uint32_t)(c / NS) & 1u;
                    if (!mbar_wait(&ctl->ready[s], ph) || *abortp) {
                        *abortp = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kb = smem_addr(smem + s * Cfg::STAGE);
                    const uint32_t vb = kb + Cfg::TILE;
                    const uint32_t lb = smem_addr(smem + Cfg::LO + (c & 1) * Cfg::TILE);
#pragma unroll
                    for (int ks = 0; ks < C / 16; ++ks) {
                        const uint32_t off = (uint32_t)ks * 2048u;   // 16 tokens = two 8-row groups
                        const uint64_t bd = smem_desc_sw128(vb + off, Cfg::BOX, 1024);
                        mma_f16(tmem, smem_desc_sw128(kb + off, Cfg::BOX, 1024), bd, idesc,
                                (j != p.jb || ks != 0) ? 1u : 0u);
                        mma_f16(tmem, smem_desc_sw128(lb + off, Cfg::BOX, 1024), bd, idesc, 1u);
                    }
                    mma_commit(&ctl->empty[s]);
                    mma_commit(&ctl->lofree[c & 1]);
                }
                if (*abortp) break;
                if (p.je > p.jb) mma_commit(&ctl->accf);   // the piece's sum is complete
                pos += advance(p);
            }
            if (*abortp) {   // drain: completes once every issued MMA is done
                mma_commit(&ctl->drain);
                mbar_wait(&ctl->drain, 0);
            }
        }
    } else {
        // ------------------------------------------------------------ key weighting + epilogue
        const int ti = threadIdx.x - 64;   // 0 .. WT-1
        const float *beta = a.beta;
        const int cp = ti & 63, rg = ti >> 6;   // diag: channel pair cp (channels 2cp, 2cp+1), row group rg
        constexpr int Q = C / 32;
        int c = 0, npiece = 0;
        for (int64_t pos = b0; pos < b1;) {
            const Piece p = piece(pos);
            const int l = p.l, h = p.h;
            const int64_t t0 = p.t0, t1 = p.t1;
            // scalar: running log-sum of the gates of the piece's tokens after the current chunk
            float rend = 0.f, rcomp = 0.f;
            float2 m = make_float2(1.f, 1.f);       // diag: product of the gates after the chunk
            float2 lam = make_float2(0.f, 0.f), lamc = make_float2(0.f, 0.f);
            float pa[Q], pb[Q];
            auto prefetch = [&](int j) {
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const int64_t t = t1 - (int64_t)(j + 1) * C + lane + 32 * q;
                    const bool v = j < p.je && t >= t0;
                    const int64_t row = ((int64_t)l * a.N + t) * a.H + h;
                    pa[q] = (!kDiag && v) ? a.alpha[row] : 1.f;
                    pb[q] = v ? (beta ? beta[row] : 1.f) : 0.f;
                }
            };
            if (warp == 2) prefetch(p.jb);
            bool ok = true;
            for (int j = p.jb; j < p.je; ++j, ++c) {
                const int s = c % NS;
                const uint32_t ph = (uint32_t)(c / NS) & 1u;
                const int par = c & 1;
                const int64_t tbase = t1 - (int64_t)(j + 1) * C;   // token of row 0 of this chunk
                if (warp == 2) {
                    if (!kDiag) {
                        float lg[Q], ex[Q];
#pragma unroll
                        for (int q = 0; q < Q; ++q) lg[q] = logf(pa[q]);   // gate is 1 outside the segment
                        float later = 0.f;   // sum over the rows above this half
#pragma unroll
                        for (int q = Q - 1; q >= 0; --q) {
                            const float inc = warp_suffix_incl(lg[q], lane);
                            ex[q] = inc - lg[q] + later;
                            later += __shfl_sync(0xffffffffu, inc, 0);
                        }
#pragma unroll
                        for (int q = 0; q < Q; ++q) ctl->rowf[par][lane + 32 * q] = pb[q] * expf(rend + ex[q]);
                        kahan(rend, rcomp, later);
                    } else {
#pragma unroll
                        for (int q = 0; q < Q; ++q) ctl->rowf[par][lane + 32 * q] = pb[q];
                    }
                    if (j + 1 < p.je) prefetch(j + 1);
                }
                ok = mbar_wait(&ctl->full[s], ph) &&
                     mbar_wait(&ctl->lofree[par], ((uint32_t)(c >> 1) & 1u) ^ 1u) && !*abortp;
                if (!bar_and(1, Cfg::WT, ok)) {
                    ok = false;
                    break;
                }
                uint8_t *kt = smem + s * Cfg::STAGE;
                uint8_t *lo = smem + Cfg::LO + par * Cfg::TILE;
                const float *rf = ctl->rowf[par];
                if (!kDiag) {
#pragma unroll
                    for (int i = 0; i < 16 * C / Cfg::WT; ++i) {
                        const int q = ti + Cfg::WT * i;          // 16-byte chunk index over both boxes
                        const int row = (q >> 3) & (C - 1);
                        uint4 hi, lw;
                        split8(*reinterpret_cast<const uint4 *>(kt + q * 16), rf[row], hi, lw);
                        *reinterpret_cast<uint4 *>(kt + q * 16) = hi;
                        *reinterpret_cast<uint4 *>(lo + q * 16) = lw;
                    }
                } else {
                    const float *at = reinterpret_cast<const float *>(kt + 2 * Cfg::TILE);
                    const int box = cp >> 5, c16 = (cp >> 2) & 7, within = (cp & 3) << 2;
                    const int r0 = rg * Cfg::RPG;
                    float2 av[Cfg::RPG];
                    float2 gp = make_float2(1.f, 1.f);
#pragma unroll
                    for (int u = 0; u < Cfg::RPG; ++u) {
                        const int r = r0 + u;
                        const bool v = tbase + r >= t0;          // rows before the segment: gate 1
                        const float2 x = *reinterpret_cast<const float2 *>(at + r * 128 + 2 * cp);
                        av[u] = v ? x : make_float2(1.f, 1.f);
                        gp.x *= av[u].x;
                        gp.y *= av[u].y;
                    }
                    ctl->gprod[par][rg][cp] = gp;
                    bar_sync(2, Cfg::WT);
                    float2 ms = m;                               // start: product over later groups
#pragma unroll
                    for (int g = Cfg::NG - 1; g >= 0; --g) {
                        const float2 pr = ctl->gprod[par][g][cp];
                        if (g > rg) {
                            ms.x *= pr.x;
                            ms.y *= pr.y;
                        }
                        m.x *= pr.x;
                        m.y *= pr.y;
                    }
                    kahan(lam.x, lamc.x, log_group(gp.x, &av[0].x, Cfg::RPG, 2));
                    kahan(lam.y, lamc.y, log_group(gp.y, &av[0].y, Cfg::RPG, 2));
#pragma unroll
                    for (int u = Cfg::RPG - 1; u >= 0; --u) {
                        const int r = r0 + u;
                        const int off = box * Cfg::BOX + r * 128 + (((c16 ^ (r & 7)) << 4) | within);
                        const uint32_t kk = *reinterpret_cast<const uint32_t *>(kt + off);
                        const float f = rf[r];                   // beta, 0 outside the segment
                        uint32_t hi, lw;
                        split2(f * ms.x * __uint_as_float(kk << 16), f * ms.y * __uint_as_float(kk & 0xFFFF0000u),
                               hi, lw);
                        *reinterpret_cast<uint32_t *>(kt + off) = hi;
                        *reinterpret_cast<uint32_t *>(lo + off) = lw;
                        ms.x *= av[u].x;
                        ms.y *= av[u].y;
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->ready[s]);
            }
            if (!ok) {
                *abortp = 1;
                break;
            }

            // -------------------------------------------------------- epilogue of the piece
            if (!bar_and(1, Cfg::WT, !*abortp)) break;   // uniform over the weighting warps
            const bool any = p.je > p.jb;
            bool ok2 = true;
            if (any) ok2 = mbar_wait(&ctl->accf, (uint32_t)npiece & 1u);
            ok2 = __all_sync(0xffffffffu, ok2);
            tc_fence_after();
            const int64_t u_out = ((int64_t)l * a.n_seg + p.seg) * a.H + h;
            float *slot = a.ws + ((int64_t)blockIdx.x * 2 + p.slot) * kSlotFloats;
            float *Sdst = p.whole ? a.S_out + u_out * 128 * 128 : slot + 128;
            const int quarter = warp & 3;               // TMEM lanes this warp may read
            const int row = quarter * 32 + lane;        // key channel = accumulator row
            constexpr int kCbPerWarp = 4 / (TW / 4);    // 32-column blocks per warp
            const int cb0 = ((warp - 2) >> 2) * kCbPerWarp;
            float *So = Sdst + (int64_t)row * 128;
#pragma unroll 1
            for (int cb = cb0; cb < cb0 + kCbPerWarp; ++cb) {
                uint32_t r[32];
                if (any && ok2) {
                    tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(cb * 32), r);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = 0u;
                }
#pragma unroll
                for (int v4 = 0; v4 < 8; ++v4)
                    reinterpret_cast<float4 *>(So + cb * 32)[v4] =
                        make_float4(__uint_as_float(r[4 * v4]), __uint_as_float(r[4 * v4 + 1]),
                                    __uint_as_float(r[4 * v4 + 2]), __uint_as_float(r[4 * v4 + 3]));
            }
            tc_fence_before();   // the accumulator's reads are done before the next piece's MMAs
            if (!ok2) *abortp = 1;
            float *ldst = p.whole ? a.lam_out + (kDiag ? u_out * 128 : u_out) : slot;
            if (kDiag) {
                ctl->lamp[rg][cp] = make_float2(lam.x - lamc.x, lam.y - lamc.y);
                bar_sync(2, Cfg::WT);
                if (rg == 0) {
                    double lx = 0.0, ly = 0.0;
                    for (int g = 0; g < Cfg::NG; ++g) {
                        lx += (double)ctl->lamp[g][cp].x;
                        ly += (double)ctl->lamp[g][cp].y;
                    }
                    reinterpret_cast<float2 *>(ldst)[cp] = make_float2((float)lx, (float)ly);
                }
                bar_sync(2, Cfg::WT);   // lamp is reused by the next piece
            } else if (ti == 0) {
                ldst[0] = (float)((double)rend - (double)rcomp);
            }
            if (any) ++npiece;
            pos += advance(p);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abortp && a.d_err) atomicExch(a.d_err, (int)HYPIC_ETIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Balanced schedule, second step: per chain, fold the partial pieces in token
// order, S <- T_p S + S_p with T_p = exp(lambda_p) (per key channel for diag),
// lambda = sum of the pieces' lambda (double); empty and invalid segments get
// lambda = 0, S = 0 (invalid ones are reported).  Eight CTAs of 128 threads per
// chain, 16 rows each; chains scanned whole by one CTA are left alone.
constexpr int kCombineParts = 8;

template <int C, bool DIAG>
__global__ void __launch_bounds__(128) sd_combine_kernel(const ScanArgs a, int G) {
    __shared__ int pre[kMaxBalSeg + 1];
    const int unit = blockIdx.x / kCombineParts, part = blockIdx.x % kCombineParts;
    const int h = unit % a.H;
    const int seg = (unit / a.H) % a.n_seg;
    const int l = unit / (a.H * a.n_seg);
    if (threadIdx.x < 32) build_prefix<C>(a, pre, threadIdx.x);
    __syncthreads();
    int64_t t0, t1;
    bool bad;
    seg_bounds(a, seg, t0, t1, bad);
    const int nc = pre[seg + 1] - pre[seg];
    const int64_t u_out = ((int64_t)l * a.n_seg + seg) * a.H + h;
    const int r = part * 16 + (threadIdx.x >> 3), c0 = (threadIdx.x & 7) * 16;   // 16 columns of row r
    float4 *S = reinterpret_cast<float4 *>(a.S_out + u_out * 128 * 128 + r * 128 + c0);
    float *lam = a.lam_out + (DIAG ? u_out * 128 : u_out);
    const bool lam_writer = DIAG ? (threadIdx.x & 7) == 0 : (part == 0 && threadIdx.x == 0);
    if (nc == 0) {
        if (bad && part == 0 && threadIdx.x == 0) flag_index_error(a.d_err);
#pragma unroll
        for (int i = 0; i < 4; ++i) S[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lam_writer) lam[DIAG ? r : 0] = 0.f;
        return;
    }
    const int64_t total = (int64_t)a.n_layers * a.H * pre[a.n_seg];
    const int64_t U0 = (int64_t)l * a.H * pre[a.n_seg] + (int64_t)a.H * pre[seg] + (int64_t)h * nc;
    const int64_t U1 = U0 + nc;
    auto owner = [&](int64_t x) { return (int)((((x + 1) * G) - 1) / total); };   // CTA whose range holds x
    auto bnd = [&](int g) { return (int64_t)g * total / G; };
    const int gf = owner(U0), gl = owner(U1 - 1);
    if (gf == gl) return;   // one CTA scanned the whole chain
    float4 acc[4];
    double lsum = 0.0;      // scalar lambda, or row r's for diag
    bool first = true;
    for (int g = gl; g >= gf; --g) {   // earliest tokens first
        if (bnd(g) == bnd(g + 1)) continue;   // a CTA with no chunks (more CTAs than chunks)
        const int slot = (g > gf || bnd(g) == U0) ? 0 : 1;
        const float *src = a.ws + ((int64_t)g * 2 + slot) * kSlotFloats;
        const float lp = DIAG ? src[r] : src[0];
        const float4 *sp = reinterpret_cast<const float4 *>(src + 128 + r * 128 + c0);
        if (first) {
            first = false;
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = sp[i];
        } else {
            const float e = expf(lp);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 v = sp[i];
                acc[i] = make_float4(fmaf(e, acc[i].x, v.x), fmaf(e, acc[i].y, v.y), fmaf(e, acc[i].z, v.z),
                                     fmaf(e, acc[i].w, v.w));
            }
        }
        lsum += (double)lp;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) S[i] = acc[i];
    if (lam_writer) lam[DIAG ? r : 0] = (float)lsum;
}

// ---------------------------------------------------------------- host side

constexpr int kMaxG = 512;   // CTAs of the balanced schedule (two per SM; scratch sized for 512)

template <int FAM, int C, int NS, int TW, bool BAL>
cudaError_t launch_tc(const ScanArgs &a, cudaStream_t s) {
    using Cfg = SdCfg<FAM, C, NS, TW>;
    const uint64_t rows = (uint64_t)a.n_layers * (uint64_t)a.N;
    CUtensorMap mk, mv, ma;
    if (!make_tensor_map_3d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k, 128, a.H, rows, 64, C,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_3d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v, 128, a.H, rows, 64, C,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (FAM == HYPIC_DIAG) {
        if (!make_tensor_map_3d(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.alpha, 128, a.H, rows, 128, C,
                                CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        ma = mk;   // unused
    }
    auto kern = scan_sd_tc_kernel<FAM, C, NS, TW, BAL>;
    constexpr int smem = sd_smem_bytes<FAM, C, NS, TW>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.n_layers * a.n_seg * a.H;
    unsigned grid = (unsigned)units;
    if (BAL) {
        int dev = 0, sms = 0;
        e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        grid = (unsigned)(2 * sms < kMaxG ? 2 * sms : kMaxG);
    }
    kern<<<grid, Cfg::THREADS, smem, s>>>(mk, mv, ma, a);
    e = cudaGetLastError();
    if (e != cudaSuccess || !BAL) return e;
    sd_combine_kernel<C, FAM == HYPIC_DIAG><<<(unsigned)(units * kCombineParts), 128, 0, s>>>(a, (int)grid);
    return cudaGetLastError();
}

}  // namespace

bool scan_sd_tc_supported(const ScanArgs &a) {
    return (a.fam == HYPIC_SCALAR || a.fam == HYPIC_DIAG) && a.in_dtype == HYPIC_BF16 && a.dk == 128 &&
           a.dv == 128 && a.o_out == nullptr && a.N > 0 && (int64_t)a.n_layers * a.N < ((int64_t)1 << 31) &&
           tensor_map_encoder() != nullptr;
}

// Diagonal gates only: their per-chunk weighting makes a CTA's own throughput the
// limit, so a grid of fewer chains than CTA slots leaves bandwidth unused (the
// balanced schedule measured 0.357 vs 0.416 ms at 8 x 8192 x 32 heads); the
// scalar scan already runs at the HBM limit with one chain per CTA (0.187 vs
// 0.192 ms before the combine step).
bool scan_sd_bal_shape(const ScanArgs &a) {
    return a.fam == HYPIC_DIAG && a.in_dtype == HYPIC_BF16 && a.dk == 128 &&
           a.dv == 128 && a.o_out == nullptr && a.N > 0 && (int64_t)a.n_layers * a.N < ((int64_t)1 << 31) &&
           a.n_seg <= kMaxBalSeg && (int64_t)a.n_layers * a.n_seg * a.H < ((int64_t)1 << 31);
}

int64_t scan_sd_bal_bytes() { return (int64_t)2 * kMaxG * kSlotFloats * 4; }

#ifndef HYPIC_SD_SCALAR_C
#define HYPIC_SD_SCALAR_C 64
#endif
#ifndef HYPIC_SD_SCALAR_NS
#define HYPIC_SD_SCALAR_NS 2
#endif
#ifndef HYPIC_SD_DIAG_C
#define HYPIC_SD_DIAG_C 32
#endif
#ifndef HYPIC_SD_DIAG_NS
#define HYPIC_SD_DIAG_NS 2
#endif
#ifndef HYPIC_SD_TW
#define HYPIC_SD_TW 8
#endif

cudaError_t launch_scan_sd_tc(const ScanArgs &a, cudaStream_t s) {
    if ((int64_t)a.n_layers * a.n_seg * a.H == 0) return cudaSuccess;
    if (a.fam == HYPIC_SCALAR)
        return launch_tc<HYPIC_SCALAR, HYPIC_SD_SCALAR_C, HYPIC_SD_SCALAR_NS, HYPIC_SD_TW, false>(a, s);
    return launch_tc<HYPIC_DIAG, HYPIC_SD_DIAG_C, HYPIC_SD_DIAG_NS, HYPIC_SD_TW, false>(a, s);
}

cudaError_t launch_scan_sd_bal(const ScanArgs &a, cudaStream_t s) {
    if ((int64_t)a.n_layers * a.n_seg * a.H == 0) return cudaSuccess;
    if (a.fam == HYPIC_SCALAR)
        return launch_tc<HYPIC_SCALAR, HYPIC_SD_SCALAR_C, HYPIC_SD_SCALAR_NS, HYPIC_SD_TW, true>(a, s);
    return launch_tc<HYPIC_DIAG, HYPIC_SD_DIAG_C, HYPIC_SD_DIAG_NS, HYPIC_SD_TW, true>(a, s);
}

}  // namespace hypic
