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
// row) are applied here; for the dense family this kernel writes the advanced
// state and the product with T_body = exp(lambda) M runs as a composition
// afterwards.
#include "internal.cuh"

namespace hypic {
namespace {

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
    constexpr int NA = FAM == HYPIC_DIAG ? DK : 1;   // gates per token
    __shared__ float sk[kTB][DK], sq[kTB][DK], sv[kTB][kCW], sa[kTB][NA], sb[kTB];
    __shared__ float red[RS][kCW];
    __shared__ float sc[FAM == HYPIC_DENSE ? 1 : DK][kCW];   // S_body slice (scalar, diag)

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
    if (FAM != HYPIC_DENSE) {
#pragma unroll
        for (int r = 0; r < 32; ++r) cp_async4(&sc[g * 32 + r][jl], a.S_C + so + (int64_t)(g * 32 + r) * DV + j);
    }
    float S[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) S[r] = a.S_prev ? a.S_prev[so + (int64_t)(g * 32 + r) * DV + j] : 0.f;

    const T *q = static_cast<const T *>(a.q), *k = static_cast<const T *>(a.k), *v = static_cast<const T *>(a.v);
    T *o = static_cast<T *>(a.o_out);
    for (int t0 = 0; t0 < a.w; t0 += kTB) {
        const int nt = a.w - t0 < kTB ? a.w - t0 : kTB;
        __syncthreads();   // the previous block's inputs are no longer read
        for (int e = tid; e < nt * DK; e += NT) {
            const int t = e / DK, c = e % DK;
            const int64_t row = (item * a.w + t0 + t) * a.H + h;   // seam token-head row
            sk[t][c] = ld_in(k, row * DK + c);
            if (o) sq[t][c] = ld_in(q, row * DK + c);
            if (FAM == HYPIC_DIAG) sa[t][c] = a.alpha[row * DK + c];
        }
        for (int e = tid; e < nt * kCW; e += NT) {
            const int t = e / kCW, c = e % kCW;
            sv[t][c] = ld_in(v, ((item * a.w + t0 + t) * a.H + h) * DV + c0 + c);
        }
        if (tid < nt) {
            const int64_t row = (item * a.w + t0 + tid) * a.H + h;
            if (FAM != HYPIC_DIAG) sa[tid][0] = a.alpha[row];
            sb[tid] = a.beta ? a.beta[row] : 1.f;
        }
        __syncthreads();
        for (int t = 0; t < nt; ++t) {
            const float b = sb[t];
            if (FAM == HYPIC_DENSE) {
                // S <- alpha (S - beta k (k^T S)) + beta k v^T = alpha S + k (beta (v - alpha u))^T, u = S^T k
                float p = 0.f;
#pragma unroll
                for (int r = 0; r < 32; ++r) p = fmaf(sk[t][g * 32 + r], S[r], p);
                red[g][jl] = p;
                __syncthreads();
                float u = 0.f;
#pragma unroll
                for (int x = 0; x < RS; ++x) u += red[x][jl];
                const float al = sa[t][0];
                const float c = b * (sv[t][jl] - al * u);
#pragma unroll
                for (int r = 0; r < 32; ++r) S[r] = fmaf(al, S[r], sk[t][g * 32 + r] * c);
                __syncthreads();   // red is reused below
            } else {
                const float bv = b * sv[t][jl];
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const float al = FAM == HYPIC_DIAG ? sa[t][g * 32 + r] : sa[t][0];
                    S[r] = fmaf(al, S[r], sk[t][g * 32 + r] * bv);
                }
            }
            if (o) {   // o_t = S_t^T q_t
                float p = 0.f;
#pragma unroll
                for (int r = 0; r < 32; ++r) p = fmaf(sq[t][g * 32 + r], S[r], p);
                red[g][jl] = p;
                __syncthreads();
                if (g == 0) {
                    float s = 0.f;
#pragma unroll
                    for (int x = 0; x < RS; ++x) s += red[x][jl];
                    o[((item * a.w + t0 + t) * a.H + h) * DV + j] = from_f32<T>(s);
                }
                __syncthreads();
            }
        }
    }

    // the rest of the segment: S_out = T_body S + S_body (dense: the advanced state only)
    if (FAM != HYPIC_DENSE) cp_async_wait_all();
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const int64_t e = so + (int64_t)(g * 32 + r) * DV + j;
        if (FAM == HYPIC_DENSE) {
            a.S_out[e] = S[r];
        } else {
            const float lam = FAM == HYPIC_DIAG ? a.lam[unit * DK + g * 32 + r] : a.lam[unit];
            a.S_out[e] = fmaf(expf(lam), S[r], sc[g * 32 + r][jl]);
        }
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
    // dense: the window in place into S_out, then S_out = exp(lambda) M S_out + S_body
    e = launch_fam<HYPIC_DENSE>(a, s);
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
