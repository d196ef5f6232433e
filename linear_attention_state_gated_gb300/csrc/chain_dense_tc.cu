// chain_dense_tc.cu -- chained composition for the gated delta rule on tcgen05.
//
// For one (request, layer, head) the combine step folds pool entries in order,
//     S <- exp(lambda_p) M_p S + S_p,
// one 128 x 128 x 128 product per step.  The product runs on the tensor cores
// in bf16 with both operands split three ways (x = hi + mid + lo, residual
// ~2^-27) and the six partial products down to order 2^-18 kept
// (~2^-26 relative per product), which keeps the fp32 composition accurate to
// well below 1e-5 at the cost of three TF32 products.  The exact fp32 running state stays in the math
// warps' registers (row i of S on TMEM lane i, two warps per lane quarter).
// Without a chain list (chain_len and seg_idx NULL) request r takes one step
// with pool entry r: the single composition S = exp(lambda) M S_prev + S_C.
// Warp 0 brings each M_p into shared memory by TMA (128-byte swizzle, so the
// row-per-lane reads are conflict-free) while the previous step's MMAs run;
// the math warps split it into TMEM as the A operand and split S into shared
// memory as the MN-major B operand; warp 1 issues the MMAs.
#include "internal.cuh"
#include "sm100.cuh"

namespace hypic {
namespace {

using namespace sm100;

constexpr int kD = 128;
constexpr int kThreads = 320;           // warp 0: TMA, warp 1: MMA, warps 2..9: math
constexpr int kMath = 256;
constexpr uint32_t kTa = 0, kTd = 256;  // TMEM: A hi / mid / lo at 0, 64, 128 (bf16 pairs); D at 256
constexpr int kBpart = 32768;           // one bf16 B tile: 128 k-rows x 128 n, 2 atoms of 64 n
constexpr int kMstage = 3 * kBpart;     // M_p, fp32, 4 boxes of 32 columns x 128 rows
constexpr int kCtl = kMstage + 65536;
constexpr int kSmem = kCtl + 1024 + 1024;

struct ChainCtrl {
    uint64_t mfull, mfree, ops_ready, d_done;
    uint32_t tmem;
    int abort;
};

// Two fp32 values -> three packed bf16 pairs with x = hi + mid + lo (to ~2^-27 relative).
__device__ __forceinline__ void split3_pair(float x0, float x1, uint32_t &hi, uint32_t &mid, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float r0 = x0 - __low2float(h), r1 = x1 - __high2float(h);
    const __nv_bfloat162 m = __floats2bfloat162_rn(r0, r1);
    const __nv_bfloat162 l = __floats2bfloat162_rn(r0 - __low2float(m), r1 - __high2float(m));
    hi = *reinterpret_cast<const uint32_t *>(&h);
    mid = *reinterpret_cast<const uint32_t *>(&m);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__global__ void __launch_bounds__(kThreads, 1)
    chain_dense_tc_kernel(const __grid_constant__ CUtensorMap tm_m, const ChainArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    ChainCtrl *ctl = reinterpret_cast<ChainCtrl *>(smem + kCtl);
    volatile int *abortp = &ctl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t u = blockIdx.x;                  // (r * Lyr + l) * H + h
    const int r = (int)(u / ((int64_t)a.n_layers * a.H));
    const int64_t lh = u % ((int64_t)a.n_layers * a.H);

    int n = a.chain_len ? a.chain_len[r] : 1;   // no list: one step, entry r (a single composition)
    if (n < 0 || n > a.max_chain) {
        if (threadIdx.x == 0) flag_index_error(a.d_err);
        n = n < 0 ? 0 : a.max_chain;
    }
    if (threadIdx.x == 0) {
        mbar_init(&ctl->mfull, 1);
        mbar_init(&ctl->mfree, kMath / 32);
        mbar_init(&ctl->ops_ready, kMath / 32);
        mbar_init(&ctl->d_done, 1);
        ctl->abort = 0;
        mbar_fence_init();
        tma_prefetch(&tm_m);
    }
    if (warp == 1) tmem_alloc(&ctl->tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;

    auto entry = [&](int c) -> int64_t {   // pool entry of step c for this layer / head
        int p = a.seg_idx ? a.seg_idx[(int64_t)r * a.max_chain + c] : r;
        if (p < 0 || p >= a.P) {
            flag_index_error(a.d_err);
            p = p < 0 ? 0 : a.P - 1;
        }
        return (int64_t)p * a.n_layers * a.H + lh;
    };

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < n; ++c) {
                if (c > 0 && (!mbar_wait(&ctl->mfree, (uint32_t)(c - 1) & 1u) || *abortp)) {
                    *abortp = 1;
                    break;
                }
                const int row = (int)(entry(c) * kD);
                mbar_expect_tx(&ctl->mfull, 65536u);
#pragma unroll
                for (int b = 0; b < 4; ++b) tma_load_3d(smem + kMstage + b * 16384, &tm_m, &ctl->mfull, 32 * b, 0, row);
                issued = c + 1;
            }
            if (*abortp && issued > 0) mbar_wait(&ctl->mfull, (uint32_t)(issued - 1) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, true);   // A TMEM, B MN-major
            const uint32_t b0 = smem_addr(smem);
            for (int c = 0; c < n; ++c) {
                if (!mbar_wait(&ctl->ops_ready, (uint32_t)c & 1u) || *abortp) {
                    *abortp = 1;
                    break;
                }
                tc_fence_after();
#pragma unroll 2
                for (int ks = 0; ks < 8; ++ks) {   // K = 128 in steps of 16 (two 8-row groups of B)
                    const uint32_t off = (uint32_t)ks * 2048u;
                    const uint64_t bh = smem_desc_sw128(b0 + off, 16384, 1024);
                    const uint64_t bm = smem_desc_sw128(b0 + kBpart + off, 16384, 1024);
                    const uint64_t bl = smem_desc_sw128(b0 + 2 * kBpart + off, 16384, 1024);
                    const uint32_t ah = tmem + kTa + (uint32_t)ks * 8u, am = ah + 64u, al = ah + 128u;
                    mma_f16_ta(tmem + kTd, ah, bh, idesc, ks > 0);
                    mma_f16_ta(tmem + kTd, ah, bm, idesc, 1u);
                    mma_f16_ta(tmem + kTd, am, bh, idesc, 1u);
                    mma_f16_ta(tmem + kTd, ah, bl, idesc, 1u);
                    mma_f16_ta(tmem + kTd, am, bm, idesc, 1u);
                    mma_f16_ta(tmem + kTd, al, bh, idesc, 1u);
                }
                mma_commit(&ctl->d_done);
            }
            if (*abortp) {
                mma_commit(&ctl->d_done);
                mbar_wait(&ctl->d_done, (uint32_t)n & 1u);
            }
        }
    } else {
        const int ch = (warp - 2) >> 2;              // column half: [64 ch, 64 ch + 64)
        const int quarter = warp & 3;
        const int i = quarter * 32 + lane;           // row of S / of M_p
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        float srow[64];                              // exact running state, row i
        {
            const float4 *init = a.S_init ? reinterpret_cast<const float4 *>(a.S_init + u * kD * kD + i * kD + ch * 64)
                                          : nullptr;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float4 v = init ? init[q] : make_float4(0.f, 0.f, 0.f, 0.f);
                srow[4 * q] = v.x; srow[4 * q + 1] = v.y; srow[4 * q + 2] = v.z; srow[4 * q + 3] = v.w;
            }
        }
        for (int c = 0; c < n; ++c) {
            const int64_t e = entry(c);
            // A = M_p (bf16 hi / mid / lo pairs) -> TMEM, row i on lane i, column k / 2
            if (!bar_and(1, kMath, mbar_wait(&ctl->mfull, (uint32_t)c & 1u) && !*abortp)) {
                *abortp = 1;
                break;
            }
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {             // 32 columns (16 packed pairs) at a time
                uint32_t hi[16], mid[16], lo[16];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int col = ch * 64 + cb * 32 + 4 * q;
                    const int box = col >> 5, chunk = (col & 31) >> 2;
                    const float4 m4 = *reinterpret_cast<const float4 *>(smem + kMstage + box * 16384 + i * 128 +
                                                                        ((chunk ^ (i & 7)) << 4));
                    split3_pair(m4.x, m4.y, hi[2 * q], mid[2 * q], lo[2 * q]);
                    split3_pair(m4.z, m4.w, hi[2 * q + 1], mid[2 * q + 1], lo[2 * q + 1]);
                }
                const uint32_t col2 = (uint32_t)(ch * 32 + cb * 16);
                tmem_st16(tmem + lane_off + kTa + col2, hi);
                tmem_st16(tmem + lane_off + kTa + 64u + col2, mid);
                tmem_st16(tmem + lane_off + kTa + 128u + col2, lo);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->mfree);     // the stage may take the next M_p
            // B = S (bf16 hi / mid / lo) -> shared memory, MN-major: row k = i, n contiguous,
            // 2 atoms of 64 columns, 128-byte swizzle
#pragma unroll
            for (int q = 0; q < 8; ++q) {                  // 8 columns (one 16-byte chunk) at a time
                const int chunk = q;                       // this thread's 64 columns are atom ch
                const int off = ch * 16384 + i * 128 + ((chunk ^ (i & 7)) << 4);
                uint32_t h[4], md[4], l[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) split3_pair(srow[8 * q + 2 * p], srow[8 * q + 2 * p + 1], h[p], md[p], l[p]);
                *reinterpret_cast<uint4 *>(smem + off) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4 *>(smem + kBpart + off) = make_uint4(md[0], md[1], md[2], md[3]);
                *reinterpret_cast<uint4 *>(smem + 2 * kBpart + off) = make_uint4(l[0], l[1], l[2], l[3]);
            }
            tmem_wait_st();
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->ops_ready);
            // this step's S_p row and decay, loaded while the MMAs run
            const float scale = expf(a.pool_lam[e]);
            const float4 *sp = reinterpret_cast<const float4 *>(a.pool_S + e * kD * kD + i * kD + ch * 64);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float4 v = __ldcs(sp + q);
                srow[4 * q] = v.x; srow[4 * q + 1] = v.y; srow[4 * q + 2] = v.z; srow[4 * q + 3] = v.w;
            }
            if (!bar_and(1, kMath, mbar_wait(&ctl->d_done, (uint32_t)c & 1u) && !*abortp)) {
                *abortp = 1;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t dv[32];
                tmem_ld32(tmem + lane_off + kTd + (uint32_t)(ch * 64 + cb * 32), dv);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 32; ++t) srow[cb * 32 + t] = fmaf(scale, __uint_as_float(dv[t]), srow[cb * 32 + t]);
            }
            tc_fence_before();
        }
        if (!*abortp) {
            float4 *out = reinterpret_cast<float4 *>(a.S_out + u * kD * kD + i * kD + ch * 64);
#pragma unroll
            for (int q = 0; q < 16; ++q)
                out[q] = make_float4(srow[4 * q], srow[4 * q + 1], srow[4 * q + 2], srow[4 * q + 3]);
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

}  // namespace

bool chain_dense_tc_supported(const ChainArgs &a) {
    return a.fam == HYPIC_DENSE && a.dk == 128 && a.dv == 128 && a.P > 0 &&
           (int64_t)a.P * a.n_layers * a.H * 128 < ((int64_t)1 << 31) && tensor_map_encoder() != nullptr;
}

cudaError_t launch_chain_dense_tc(const ChainArgs &a, cudaStream_t s) {
    const int64_t units = (int64_t)a.R * a.n_layers * a.H;
    if (units == 0) return cudaSuccess;
    CUtensorMap tm;
    const uint64_t rows = (uint64_t)a.P * a.n_layers * a.H * 128;
    if (!make_tensor_map_3d(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.pool_M, 128, 1, rows, 32, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(chain_dense_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    chain_dense_tc_kernel<<<(unsigned)units, kThreads, kSmem, s>>>(tm, a);
    return cudaGetLastError();
}

}  // namespace hypic
