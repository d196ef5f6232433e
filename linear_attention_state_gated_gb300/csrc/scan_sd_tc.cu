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
// Per CTA one (layer, segment, head) chain, d_k = d_v = 128:
//   warp 0     TMA producer: K, V (and the diagonal gates) of a chunk of C
//              tokens into a ring of NS shared-memory stages (128B swizzle);
//   warps 2-5  weight the keys: K~ = w * beta * k, split exactly into
//              bf16 hi + lo (K~ - hi), written over K / into a lo tile in the
//              same swizzled positions; later the epilogue (TMEM -> S);
//   warp 1     one thread issues tcgen05.mma: D[128x128] += K~hi^T V + K~lo^T V
//              (both operands MN-major, M = key channel, N = value channel,
//              K = token), commits each stage back to the producer.
// V is used exactly (bf16 input); the hi/lo split keeps K~ to ~2^-17 relative.
// Every wait is time-bounded; a timeout is reported as HYPIC_ETIMEOUT.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "sm100.cuh"

namespace hypic {
namespace {

using namespace sm100;

constexpr int kThreads = 192;
constexpr int kTmemCols = 128;

template <int FAM, int C, int NS>
struct SdCfg {
    static constexpr int BOX = C * 128;                    // 64 channels x C tokens, bf16
    static constexpr int TILE = 2 * BOX;                   // 128 channels
    static constexpr int ATILE = FAM == HYPIC_DIAG ? C * 512 : 0;   // fp32 gates
    static constexpr int STAGE = 2 * TILE + ATILE;         // TMA ring stage: K (-> K~hi), V, gates
    static constexpr uint32_t TX = STAGE;                  // bytes TMA brings per stage
    static constexpr int LO = NS * STAGE;                  // two K~lo tiles (chunk parity) after the ring
    static constexpr int SMEM = NS * STAGE + 2 * TILE + 2048;   // + control block + alignment slack
    static_assert(C == 32 || C == 64, "chunk of 32 or 64 tokens");
    static_assert(NS >= 2 && NS <= 8, "2 to 8 stages");
    static_assert(STAGE % 1024 == 0, "stages stay 1024-byte aligned");
};

struct SdCtrl {
    uint64_t full[8], ready[8], empty[8], lofree[2], accf;
    float rowf[2][64];
    uint32_t tmem;
    int abort;
};

__device__ __forceinline__ float warp_suffix_incl(float x, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, x, off);
        if (lane + off < 32) x += y;
    }
    return x;
}

__device__ __forceinline__ void split8(const uint4 raw, const float w, uint4 &hi, uint4 &lo) {
    const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t h[4], l[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float x0 = __uint_as_float(in[p] << 16) * w;
        const float x1 = __uint_as_float(in[p] & 0xFFFF0000u) * w;
        const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
        const float r0 = x0 - __low2float(hh), r1 = x1 - __high2float(hh);
        const __nv_bfloat162 ll = __floats2bfloat162_rn(r0, r1);
        h[p] = *reinterpret_cast<const uint32_t *>(&hh);
        l[p] = *reinterpret_cast<const uint32_t *>(&ll);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ float pow2f(int e) {   // 2^e, 0 below the normal range
    return e < -126 ? 0.f : __int_as_float((e + 127) << 23);
}

template <int FAM, int C, int NS>
__global__ void __launch_bounds__(kThreads, 1)
    scan_sd_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_a, const ScanArgs a) {
    using Cfg = SdCfg<FAM, C, NS>;
    constexpr bool kDiag = FAM == HYPIC_DIAG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    SdCtrl *ctl = reinterpret_cast<SdCtrl *>(smem + Cfg::LO + 2 * Cfg::TILE);
    volatile int *abortp = &ctl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int unit = blockIdx.x;
    const int h = unit % a.H;
    const int seg = (unit / a.H) % a.n_seg;
    const int l = unit / (a.H * a.n_seg);
    int64_t t0 = a.seg_offsets[seg], t1 = a.seg_offsets[seg + 1];
    const bool bad = !(t0 >= 0 && t0 <= t1 && t1 <= a.N);
    if (bad) t0 = t1 = 0;
    const int nc = (int)((t1 - t0 + C - 1) / C);
    const int64_t row_end = (int64_t)l * a.N + t1;   // token row just past the segment

    if (threadIdx.x == 0) {
        if (bad) flag_index_error(a.d_err);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->ready[s], 4);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->lofree[0], 1);
        mbar_init(&ctl->lofree[1], 1);
        mbar_init(&ctl->accf, 1);
        ctl->abort = 0;
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(&ctl->tmem, kTmemCols);
    if (threadIdx.x == 32 * 0) {
        tma_prefetch(&tm_k);
        tma_prefetch(&tm_v);
        if (kDiag) tma_prefetch(&tm_a);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            for (int j = 0; j < nc; ++j) {
                const int s = j % NS;
                const uint32_t ph = (uint32_t)(j / NS) & 1u;
                if (!mbar_wait(&ctl->empty[s], ph ^ 1u) || *abortp) {
                    *abortp = 1;
                    break;
                }
                uint8_t *st = smem + s * Cfg::STAGE;
                const int row = (int)(row_end - (int64_t)(j + 1) * C);
                mbar_expect_tx(&ctl->full[s], Cfg::TX);
                tma_load_3d(st, &tm_k, &ctl->full[s], 0, h, row);
                tma_load_3d(st + Cfg::BOX, &tm_k, &ctl->full[s], 64, h, row);
                tma_load_3d(st + Cfg::TILE, &tm_v, &ctl->full[s], 0, h, row);
                tma_load_3d(st + Cfg::TILE + Cfg::BOX, &tm_v, &ctl->full[s], 64, h, row);
                if (kDiag) tma_load_3d(st + 2 * Cfg::TILE, &tm_a, &ctl->full[s], 0, h, row);
                issued = j + 1;
            }
            if (*abortp) {   // let copies already in flight land before the CTA leaves
                for (int j = issued - NS < 0 ? 0 : issued - NS; j < issued; ++j)
                    mbar_wait(&ctl->full[j % NS], (uint32_t)(j / NS) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 128, true, true);
            for (int j = 0; j < nc; ++j) {
                const int s = j % NS;
                const uint32_t ph = (uint32_t)(j / NS) & 1u;
                if (!mbar_wait(&ctl->ready[s], ph) || *abortp) {
                    *abortp = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t kb = smem_addr(smem + s * Cfg::STAGE);
                const uint32_t vb = kb + Cfg::TILE;
                const uint32_t lb = smem_addr(smem + Cfg::LO + (j & 1) * Cfg::TILE);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks) {
                    const uint32_t off = (uint32_t)ks * 2048u;   // 16 tokens = two 8-row groups
                    const uint64_t bd = smem_desc_sw128(vb + off, Cfg::BOX, 1024);
                    mma_f16(tmem, smem_desc_sw128(kb + off, Cfg::BOX, 1024), bd, idesc, (j | ks) != 0);
                    mma_f16(tmem, smem_desc_sw128(lb + off, Cfg::BOX, 1024), bd, idesc, 1u);
                }
                mma_commit(&ctl->empty[s]);
                mma_commit(&ctl->lofree[j & 1]);
            }
            if (nc > 0) {
                mma_commit(&ctl->accf);
                if (*abortp) mbar_wait(&ctl->accf, 0);
            }
        }
    } else {
        // ------------------------------------------------------------ key weighting
        const int ti = threadIdx.x - 64;   // 0..127
        const float *beta = a.beta;
        // scalar: running log-sum of the gates of tokens after the current chunk
        float rend = 0.f, rcomp = 0.f;
        // diag: running product of later gates for channel ti, as m * 2^E
        float m = 1.f, scale = 1.f;
        int E = 0;
        constexpr int Q = C / 32;
        float pa[Q], pb[Q];
        auto prefetch = [&](int j) {
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const int64_t t = t1 - (int64_t)(j + 1) * C + lane + 32 * q;
                const bool v = j < nc && t >= t0;
                const int64_t row = ((int64_t)l * a.N + t) * a.H + h;
                pa[q] = (!kDiag && v) ? a.alpha[row] : 1.f;
                pb[q] = v ? (beta ? beta[row] : 1.f) : 0.f;
            }
        };
        if (warp == 2) prefetch(0);

        for (int j = 0; j < nc; ++j) {
            const int s = j % NS;
            const uint32_t ph = (uint32_t)(j / NS) & 1u;
            const int par = j & 1;
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
                    // Kahan-compensated running sum of the chunk totals
                    const float y = later - rcomp;
                    const float t = rend + y;
                    rcomp = (t - rend) - y;
                    rend = t;
                } else {
#pragma unroll
                    for (int q = 0; q < Q; ++q) ctl->rowf[par][lane + 32 * q] = pb[q];
                }
                if (j + 1 < nc) prefetch(j + 1);
            }
            const bool ok = mbar_wait(&ctl->full[s], ph) &&
                            mbar_wait(&ctl->lofree[par], ((uint32_t)(j >> 1) & 1u) ^ 1u) && !*abortp;
            if (!bar_and(1, 128, ok)) {
                *abortp = 1;
                break;
            }
            uint8_t *kt = smem + s * Cfg::STAGE;
            uint8_t *lo = smem + Cfg::LO + par * Cfg::TILE;
            if (!kDiag) {
#pragma unroll 4
                for (int i = 0; i < 16 * C / 128; ++i) {
                    const int q = ti + 128 * i;             // 16-byte chunk index over both boxes
                    const int row = (q >> 3) & (C - 1);
                    const float w = ctl->rowf[par][row];
                    uint4 hi, lw;
                    split8(*reinterpret_cast<const uint4 *>(kt + q * 16), w, hi, lw);
                    *reinterpret_cast<uint4 *>(kt + q * 16) = hi;
                    *reinterpret_cast<uint4 *>(lo + q * 16) = lw;
                }
            } else {
                const float *at = reinterpret_cast<const float *>(kt + 2 * Cfg::TILE);
                const int box = ti >> 6, ci = ti & 63, c16 = ci >> 3, within = ci & 7;
                const float *rf = ctl->rowf[par];
                // rows in groups of 8, last row first: all loads of a group are
                // issued before the sequential product over its rows
#pragma unroll
                for (int g = C / 8 - 1; g >= 0; --g) {
                    float av[8], kv[8];
                    int offs[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int r = 8 * g + u;
                        offs[u] = box * Cfg::BOX + r * 128 + (((c16 ^ (r & 7)) << 4) | (within << 1));
                        av[u] = at[r * 128 + ti];
                        kv[u] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(kt + offs[u]));
                    }
#pragma unroll
                    for (int u = 7; u >= 0; --u) {
                        const int r = 8 * g + u;
                        const bool v = tbase + r >= t0;          // rows before the segment add nothing
                        const float x = rf[r] * (m * scale) * kv[u];   // rf = beta (0 outside)
                        const __nv_bfloat16 xh = __float2bfloat16_rn(x);
                        *reinterpret_cast<__nv_bfloat16 *>(kt + offs[u]) = xh;
                        *reinterpret_cast<__nv_bfloat16 *>(lo + offs[u]) =
                            __float2bfloat16_rn(x - __bfloat162float(xh));
                        m *= v ? av[u] : 1.f;
                        if (m < 0x1p-60f) {
                            m *= 0x1p64f;
                            E -= 64;
                            scale = pow2f(E);
                        }
                    }
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->ready[s]);
        }

        // ------------------------------------------------------------ epilogue
        const int64_t u_out = ((int64_t)l * a.n_seg + seg) * a.H + h;
        if (!*abortp) {
            bool ok = true;
            if (nc > 0) ok = mbar_wait(&ctl->accf, 0);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            const int quarter = warp & 3;               // TMEM lanes this warp may read
            const int row = quarter * 32 + lane;        // key channel = accumulator row
            float *So = a.S_out + u_out * 128 * 128 + (int64_t)row * 128;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t r[32];
                if (nc > 0 && ok) {
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
            if (!ok) *abortp = 1;
            if (kDiag) {
                const double lam = (double)logf(m) + (double)E * 0.69314718055994530942;
                a.lam_out[u_out * 128 + ti] = (float)lam;
            } else if (ti == 0) {
                a.lam_out[u_out] = (float)((double)rend - (double)rcomp);
            }
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

// ---------------------------------------------------------------- host side

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

// 3-D map over [rows][H][inner] with box {box0, 1, box2}.
bool make_map(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *base, uint64_t inner, uint64_t H,
              uint64_t rows, uint32_t box0, uint32_t box2, CUtensorMapSwizzle sw) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {inner, H, rows};
    const cuuint64_t strides[2] = {inner * esize, inner * H * esize};
    const cuuint32_t box[3] = {box0, 1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FAM, int C, int NS>
cudaError_t launch_tc(const ScanArgs &a, cudaStream_t s) {
    using Cfg = SdCfg<FAM, C, NS>;
    const uint64_t rows = (uint64_t)a.n_layers * (uint64_t)a.N;
    CUtensorMap mk, mv, ma;
    if (!make_map(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k, 128, a.H, rows, 64, C,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v, 128, a.H, rows, 64, C,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (FAM == HYPIC_DIAG) {
        if (!make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.alpha, 128, a.H, rows, 128, C,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        ma = mk;   // unused
    }
    auto kern = scan_sd_tc_kernel<FAM, C, NS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.n_layers * a.n_seg * a.H;
    kern<<<(unsigned)units, kThreads, Cfg::SMEM, s>>>(mk, mv, ma, a);
    return cudaGetLastError();
}

}  // namespace

bool scan_sd_tc_supported(const ScanArgs &a) {
    return (a.fam == HYPIC_SCALAR || a.fam == HYPIC_DIAG) && a.in_dtype == HYPIC_BF16 && a.dk == 128 &&
           a.dv == 128 && a.o_out == nullptr && a.N > 0 && (int64_t)a.n_layers * a.N < ((int64_t)1 << 31) &&
           encode_fn() != nullptr;
}

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

cudaError_t launch_scan_sd_tc(const ScanArgs &a, cudaStream_t s) {
    if ((int64_t)a.n_layers * a.n_seg * a.H == 0) return cudaSuccess;
    if (a.fam == HYPIC_SCALAR) return launch_tc<HYPIC_SCALAR, HYPIC_SD_SCALAR_C, HYPIC_SD_SCALAR_NS>(a, s);
    return launch_tc<HYPIC_DIAG, HYPIC_SD_DIAG_C, HYPIC_SD_DIAG_NS>(a, s);
}

}  // namespace hypic
