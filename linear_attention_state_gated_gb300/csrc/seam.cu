// seam.cu -- seam-window advance fused with the composition of the rest of a
// reused segment.
//
// xix.ai/fr, paragraph on full-attention layers ("fenetres de jonction"): the
// first w tokens of every reused segment are not cached; at reuse they are
// recomputed under the full prefix, the linear layers advance the running state
// through them and hand each seam token's output to the layer above, and the
// rest of the segment enters through its cached pair (T_body, S_body).  Per item
// and head:
//   S = S_prev;  for t < w:  S = T_t S + beta_t k_t v_t^T,  o_t = S^T q_t;
//   S_out = T_body S + S_body.
//
// Every step of the window acts on each column of S on its own (for the gated
// delta rule too: u_j = k^T S e_j, then column j's rank-one update and output
// entry), so one CTA takes a 32-column slice of one (item, head): thread (j, g)
// owns column j of the slice over rows 32 g .. 32 g + 31 in registers (fp32).
// Each warp reads and writes 128-byte row pieces, and many small CTAs per SM keep
// the state traffic in flight.  The reductions over rows a token needs (k^T S for
// the gated delta rule, S^T q for the output) go through shared memory across
// the row groups.  The window's inputs are staged in shared memory a block of
// tokens at a time.  Scalar and diagonal T_body (exp(lambda) per head or per
// row) are applied here; for the dense and KDA families (the latter a gate per
// channel inside the erasing update) this kernel writes the advanced state and
// the product with T_body = exp(lambda) M runs as a composition afterwards.
#include "internal.cuh"
#include "sm100.cuh"

namespace hypic {
namespace {

using namespace sm100;

constexpr int kTB = 8;   // seam tokens staged per block

template <typename T>
__device__ __forceinline__ float ld_in(const T *p, int64_t i) {
    return to_f32(p[i]);
}

// 4-byte asynchronous global -> shared copy (completes at cp_async_wait_all)
__device__ __forceinline__ void cp_async4(float *dst, const float *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

constexpr int kCW = 32;   // columns of S per CTA

template <int FAM, int DK, int DV, typename T>
__global__ void __launch_bounds__(kCW *(DK / 32)) seam_kernel(const SeamArgs a) {
    constexpr int RS = DK / 32;               // row groups
    constexpr int NT = kCW * RS;
    constexpr int NS = DV / kCW;              // column slices per (item, head)
    constexpr bool kDelta = FAM == HYPIC_DENSE || FAM == HYPIC_KDA;   // erasing update, operator exp(lambda) M
    constexpr bool kGateRow = FAM == HYPIC_DIAG || FAM == HYPIC_KDA;  // a gate per channel
    constexpr int NA = kGateRow ? DK : 1;            // gates per token
    __shared__ float sk[kTB][DK], sq[kTB][DK], sv[kTB][kCW], sa[kTB][NA], sb[kTB];
    __shared__ float red[2][RS][kCW];                        // S^T k partials, by token parity
    __shared__ float ro[RS][kTB][kCW];                       // output partials of a block of tokens
    __shared__ float sc[kDelta ? 1 : DK][kCW];               // S_body slice (scalar, diag)
    __shared__ float sl[FAM == HYPIC_DIAG ? DK : 1];         // exp(lambda_body) per row (diag)

    const int tid = threadIdx.x;
    const int jl = tid % kCW, g = tid / kCW;  // column in the slice, row group
    const int64_t unit = blockIdx.x / NS;     // item * H + head
    const int c0 = (int)(blockIdx.x % NS) * kCW;
    const int j = c0 + jl;                    // column of S
    const int64_t item = unit / a.H;
    const int h = (int)(unit % a.H);
    const int64_t so = unit * DK * DV;

    // S_body's slice starts on its way to shared memory now, so its latency overlaps
    // the window (each thread copies, and later reads, its own elements)
    if (!kDelta) {
#pragma unroll
        for (int r = 0; r < 32; ++r) cp_async4(&sc[g * 32 + r][jl], a.S_C + so + (int64_t)(g * 32 + r) * DV + j);
    }
    float S[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) S[r] = a.S_prev ? a.S_prev[so + (int64_t)(g * 32 + r) * DV + j] : 0.f;

    if (FAM == HYPIC_DIAG)
        for (int r = tid; r < DK; r += NT) sl[r] = expf(a.lam[unit * DK + r]);

    const T *q = static_cast<const T *>(a.q), *k = static_cast<const T *>(a.k), *v = static_cast<const T *>(a.v);
    T *o = static_cast<T *>(a.o_out);
    for (int t0 = 0; t0 < a.w; t0 += kTB) {
        const int nt = a.w - t0 < kTB ? a.w - t0 : kTB;
        __syncthreads();   // the previous block's inputs and output partials are no longer read
        for (int e = tid; e < nt * DK; e += NT) {
            const int t = e / DK, c = e % DK;
            const int64_t row = (item * a.w + t0 + t) * a.H + h;   // seam token-head row
            sk[t][c] = ld_in(k, row * DK + c);
            if (o) sq[t][c] = ld_in(q, row * DK + c);
            if (kGateRow) sa[t][c] = a.alpha[row * DK + c];
        }
        for (int e = tid; e < nt * kCW; e += NT) {
            const int t = e / kCW, c = e % kCW;
            sv[t][c] = ld_in(v, ((item * a.w + t0 + t) * a.H + h) * DV + c0 + c);
        }
        if (tid < nt) {
            const int64_t row = (item * a.w + t0 + tid) * a.H + h;
            if (!kGateRow) sa[tid][0] = a.alpha[row];
            sb[tid] = a.beta ? a.beta[row] : 1.f;
        }
        __syncthreads();
        float po[kTB];   // this thread's partial outputs (its 32 rows) of the block's tokens
#pragma unroll
        for (int t = 0; t < kTB; ++t) {
            if (t < nt) {
                const float b = sb[t];
                const float *kt = &sk[t][g * 32];
                float c;   // S <- alpha S + k c^T, column entry c_j
                float nbu = 0.f;   // KDA: -beta u_j (the erasure, before the per-row gate)
                if (kDelta) {
                    // gated delta rule: c = beta (v - alpha u), u = S^T k (rows summed over the groups)
                    uint64_t p2 = 0;
#pragma unroll
                    for (int rq = 0; rq < 8; ++rq) {
                        const float4 k4 = *reinterpret_cast<const float4 *>(kt + 4 * rq);
                        p2 = fma2(pk2(k4.x, k4.y), pk2(S[4 * rq], S[4 * rq + 1]), p2);
                        p2 = fma2(pk2(k4.z, k4.w), pk2(S[4 * rq + 2], S[4 * rq + 3]), p2);
                    }
                    float plo, phi;
                    upk2(p2, plo, phi);
                    red[t & 1][g][jl] = plo + phi;
                    __syncthreads();   // (red alternates by token, so one barrier a token suffices)
                    float u = 0.f;
#pragma unroll
                    for (int x = 0; x < RS; ++x) u += red[t & 1][x][jl];
                    if (FAM == HYPIC_DENSE) {
                        c = b * (sv[t][jl] - sa[t][0] * u);
                    } else {   // KDA: S <- diag(alpha) (S - beta k u^T) + beta k v^T
                        c = b * sv[t][jl];
                        nbu = -b * u;
                    }
                } else {
                    c = b * sv[t][jl];
                }
                const uint64_t cc = pk2(c, c);
#pragma unroll
                for (int rq = 0; rq < 8; ++rq) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(kt + 4 * rq);
                    uint64_t a01, a23;
                    if (kGateRow) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(&sa[t][g * 32 + 4 * rq]);
                        a01 = pk2(a4.x, a4.y);
                        a23 = pk2(a4.z, a4.w);
                    } else {
                        a01 = a23 = pk2(sa[t][0], sa[t][0]);
                    }
                    uint64_t x01 = pk2(S[4 * rq], S[4 * rq + 1]), x23 = pk2(S[4 * rq + 2], S[4 * rq + 3]);
                    if (FAM == HYPIC_KDA) {   // the erasure first, then the per-row gate
                        const uint64_t nb = pk2(nbu, nbu);
                        x01 = fma2(pk2(k4.x, k4.y), nb, x01);
                        x23 = fma2(pk2(k4.z, k4.w), nb, x23);
                    }
                    const uint64_t s01 = fma2(a01, x01, mul2(pk2(k4.x, k4.y), cc));
                    const uint64_t s23 = fma2(a23, x23, mul2(pk2(k4.z, k4.w), cc));
                    upk2(s01, S[4 * rq], S[4 * rq + 1]);
                    upk2(s23, S[4 * rq + 2], S[4 * rq + 3]);
                }
                if (o) {   // this thread's part of o_t = S_t^T q_t
                    const float *qt = &sq[t][g * 32];
                    uint64_t p2 = 0;
#pragma unroll
                    for (int rq = 0; rq < 8; ++rq) {
                        const float4 q4 = *reinterpret_cast<const float4 *>(qt + 4 * rq);
                        p2 = fma2(pk2(q4.x, q4.y), pk2(S[4 * rq], S[4 * rq + 1]), p2);
                        p2 = fma2(pk2(q4.z, q4.w), pk2(S[4 * rq + 2], S[4 * rq + 3]), p2);
                    }
                    float plo, phi;
                    upk2(p2, plo, phi);
                    po[t] = plo + phi;
                }
            }
        }
        if (o) {   // the block's outputs: row groups summed once for all its tokens
#pragma unroll
            for (int t = 0; t < kTB; ++t)
                if (t < nt) ro[g][t][jl] = po[t];
            __syncthreads();
            if (g == 0) {
                for (int t = 0; t < nt; ++t) {
                    float sum = 0.f;
#pragma unroll
                    for (int x = 0; x < RS; ++x) sum += ro[x][t][jl];
                    o[((item * a.w + t0 + t) * a.H + h) * DV + j] = from_f32<T>(sum);
                }
            }
        }
    }

    // the rest of the segment: S_out = T_body S + S_body (dense: the advanced state only)
    if (!kDelta) cp_async_wait_all();
    if (FAM == HYPIC_DIAG) __syncthreads();   // sl is in (also without a window)
    const float el = FAM == HYPIC_SCALAR ? expf(a.lam[unit]) : 1.f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const int64_t e = so + (int64_t)(g * 32 + r) * DV + j;
        if (kDelta)
            a.S_out[e] = S[r];
        else
            a.S_out[e] = fmaf(FAM == HYPIC_DIAG ? sl[g * 32 + r] : el, S[r], sc[g * 32 + r][jl]);
    }
}

template <int FAM, int DK, int DV>
cudaError_t launch_typed(const SeamArgs &a, cudaStream_t s) {
    const unsigned grid = (unsigned)((int64_t)a.n * a.H * (DV / kCW));
    if (a.in_dtype == HYPIC_BF16)
        seam_kernel<FAM, DK, DV, __nv_bfloat16><<<grid, kCW * (DK / 32), 0, s>>>(a);
    else
        seam_kernel<FAM, DK, DV, float><<<grid, kCW * (DK / 32), 0, s>>>(a);
    return cudaGetLastError();
}

template <int FAM>
cudaError_t launch_fam(const SeamArgs &a, cudaStream_t s) {
#define HYPIC_SEAM_DD(K, V) \
    if (a.dk == K && a.dv == V) return launch_typed<FAM, K, V>(a, s);
    HYPIC_SEAM_DD(32, 32) HYPIC_SEAM_DD(32, 64) HYPIC_SEAM_DD(32, 128)
    HYPIC_SEAM_DD(64, 32) HYPIC_SEAM_DD(64, 64) HYPIC_SEAM_DD(64, 128)
    HYPIC_SEAM_DD(128, 32) HYPIC_SEAM_DD(128, 64) HYPIC_SEAM_DD(128, 128)
#undef HYPIC_SEAM_DD
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_seam_compose(const SeamArgs &a, cudaStream_t s) {
    if ((int64_t)a.n * a.H == 0) return cudaSuccess;
    cudaError_t e;
    if (a.fam == HYPIC_SCALAR) return launch_fam<HYPIC_SCALAR>(a, s);
    if (a.fam == HYPIC_DIAG) return launch_fam<HYPIC_DIAG>(a, s);
    // dense, KDA: the window in place into S_out, then S_out = exp(lambda) M S_out + S_body
    e = a.fam == HYPIC_KDA ? launch_fam<HYPIC_KDA>(a, s) : launch_fam<HYPIC_DENSE>(a, s);
    if (e != cudaSuccess) return e;
    ComposeArgs c{};
    c.fam = HYPIC_DENSE;
    c.n = a.n;
    c.H = a.H;
    c.dk = a.dk;
    c.dv = a.dv;
    c.lam = a.lam;
    c.M = a.M;
    c.S_prev = a.S_out;
    c.S_C = a.S_C;
    c.S_out = a.S_out;
    return launch_compose(c, s);
}

}  // namespace hypic
