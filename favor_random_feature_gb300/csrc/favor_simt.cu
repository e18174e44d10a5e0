// favor_simt.cu -- the fp32 SIMT path: FAVOR+ forward in FFMA with accurate
// expf / sincosf.  It serves the fp32 entry point (favor_attn_forward_f32),
// the standalone feature map, and bf16 shapes the tensor-core path does not
// cover.  Every step runs on the GPU.
//
// Steps (one head = one (b, h)):
//   1. projections   P[t][n] = w_n . x_t                     (omega rows w_n)
//   2. features      positive: phi~ = exp(P - max_n P), row log-scale
//                              c - |x|^2/2 - ln(m)/2 (exact feature = phi~ e^logscale)
//                    trig:     (sin P_n, cos P_n), log-scale -ln(m)/2
//                    elu1:     P = x, phi = x+1 | e^x, log-scale 0
//      -- "Kernel Feature Maps" sections 1, 3, 4; Performer page, phi(x).
//   3. key weights   phi_K <- phi~_K * exp(logscale_j - max_j logscale_j):
//      one per-head constant factor, which cancels in the ratio.
//   4a. non-causal   KVz = phi_K^T [V | 1]; out = phi~_Q KV / phi~_Q z
//      -- Performer page In[25]; study notes "Core points" steps 4-5.
//   4b. causal       per 64-row chunk the state entering it (the sum of the
//      chunk states phi_K(c)^T [V_c | 1] before it); out_i = (phi_q S_in +
//      sum_{j<=i in chunk} A_ij v_j) / (phi_q z_in + sum_{j<=i} A_ij),
//      A_ij = phi~_q_i . phi_K_j -- study notes "Case 2" (prefix sum),
//      diagonal included.
//   Steps 4a/4b run on state_scan and chunk_rows, the kernels the backward
//   pass uses too.
#include <cmath>

#include <cuda_bf16.h>

#include "favor_internal.h"

namespace favor {
namespace {

__device__ __forceinline__ float load_in(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_in(const uint16_t *p, size_t i) {
    return __uint_as_float(static_cast<uint32_t>(p[i]) << 16);
}
// four consecutive input elements (i % 4 == 0; 16-byte fp32 or 8-byte bf16 loads)
__device__ __forceinline__ float4 load4_in(const float *p, size_t i) { return *reinterpret_cast<const float4 *>(p + i); }
__device__ __forceinline__ float4 load4_in(const uint16_t *p, size_t i) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p + i);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
}
// the bits of four consecutive input elements (i % 4 == 0), converted later
// (a prefetch that converts at once waits for its load there)
__device__ __forceinline__ uint4 load4_raw(const float *p, size_t i) { return *reinterpret_cast<const uint4 *>(p + i); }
__device__ __forceinline__ uint4 load4_raw(const uint16_t *p, size_t i) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p + i);
    return make_uint4(u.x, u.y, 0u, 0u);
}
template <typename T>
__device__ __forceinline__ float4 from_raw4(uint4 b) {
    if (sizeof(T) == 4) return make_float4(__uint_as_float(b.x), __uint_as_float(b.y), __uint_as_float(b.z), __uint_as_float(b.w));
    return make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xffff0000u), __uint_as_float(b.y << 16),
                       __uint_as_float(b.y & 0xffff0000u));
}
__device__ __forceinline__ void store_out(float *p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, size_t i, float v) { p[i] = __float2bfloat16_rn(v); }

// Register-tiled products of shared-memory tiles for 16 RS threads, ty = tid / 16,
// tx = tid % 16.  A thread owns rows ty + RS u (u < RU, RS RU = 64) of the result
// and the columns 4 tx + w (mm_nn) or tx + 16 w (mm_nt), w < 4; the operands are
// read 4 values of the contraction at a time (16-byte loads: RU + 4 loads per
// 16 RU FMAs).
// Row pitches are multiples of 4 floats; the B rows that 16 threads read at once
// (mm_nt) have an odd pitch in 16-byte units, so those loads do not conflict.
//   mm_nn: acc[u][w] += sum_k A[ty + RS u][k] B[k][4 tx + w]
//   mm_nt: acc[u][w] += sum_k A[ty + RS u][k] B[tx + 16 w][k]
// With BLK the rows are 4 ty + u instead (the A rows a warp reads are still
// shared by its 16-thread halves), so that a triangular operand's loop can
// stop at the diagonal (k0, k1: the contraction range, multiples of 4).
template <int RU = 4, int RS = 16, bool BLK = false>
__device__ __forceinline__ void mm_nn(float (&acc)[RU][4], const float *A, int lda, const float *B, int ldb, int K,
                                      int ty, int tx, int k0 = 0) {
#pragma unroll 2
    for (int k = k0; k < K; k += 4) {
        float4 a[RU], b[4];
#pragma unroll
        for (int u = 0; u < RU; ++u)
            a[u] = *reinterpret_cast<const float4 *>(A + (BLK ? RU * ty + u : ty + RS * u) * lda + k);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) b[kk] = *reinterpret_cast<const float4 *>(B + (k + kk) * ldb + 4 * tx);
#pragma unroll
        for (int u = 0; u < RU; ++u) {
            const float av[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                acc[u][0] = fmaf(av[kk], b[kk].x, acc[u][0]);
                acc[u][1] = fmaf(av[kk], b[kk].y, acc[u][1]);
                acc[u][2] = fmaf(av[kk], b[kk].z, acc[u][2]);
                acc[u][3] = fmaf(av[kk], b[kk].w, acc[u][3]);
            }
        }
    }
}

template <int RU = 4, int RS = 16, bool BLK = false>
__device__ __forceinline__ void mm_nt(float (&acc)[RU][4], const float *A, int lda, const float *B, int ldb, int K,
                                      int ty, int tx) {
#pragma unroll 2
    for (int k = 0; k < K; k += 4) {
        float4 a[RU], b[4];
#pragma unroll
        for (int u = 0; u < RU; ++u)
            a[u] = *reinterpret_cast<const float4 *>(A + (BLK ? RU * ty + u : ty + RS * u) * lda + k);
#pragma unroll
        for (int w = 0; w < 4; ++w) b[w] = *reinterpret_cast<const float4 *>(B + (tx + 16 * w) * ldb + k);
#pragma unroll
        for (int u = 0; u < RU; ++u)
#pragma unroll
            for (int w = 0; w < 4; ++w)
                acc[u][w] = fmaf(a[u].x, b[w].x,
                                 fmaf(a[u].y, b[w].y, fmaf(a[u].z, b[w].z, fmaf(a[u].w, b[w].w, acc[u][w]))));
    }
}

// acc[u][w] += sum_k A[k][ty + 16 u] B[k][4 tx + w] (BLK: A[k][4 ty + u]), k
// in [k0, K): both operands row-major with the contraction along their rows
// (4 broadcast scalar loads, or one 16-byte load with BLK, and one 16-byte
// load per 16 FMAs)
template <bool BLK = false>
__device__ __forceinline__ void mm_tn(float (&acc)[4][4], const float *A, int lda, const float *B, int ldb, int K,
                                      int ty, int tx, int k0 = 0) {
#pragma unroll 4
    for (int k = k0; k < K; ++k) {
        float a[4];
        if (BLK) {
            const float4 a4 = *reinterpret_cast<const float4 *>(A + k * lda + 4 * ty);
            a[0] = a4.x, a[1] = a4.y, a[2] = a4.z, a[3] = a4.w;
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) a[u] = A[k * lda + ty + 16 * u];
        }
        const float4 b = *reinterpret_cast<const float4 *>(B + k * ldb + 4 * tx);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            acc[u][0] = fmaf(a[u], b.x, acc[u][0]);
            acc[u][1] = fmaf(a[u], b.y, acc[u][1]);
            acc[u][2] = fmaf(a[u], b.z, acc[u][2]);
            acc[u][3] = fmaf(a[u], b.w, acc[u][3]);
        }
    }
}

// 1. projections P[t][n] = w_n . x_t: block = 64 tokens x 64 projections of
// one head, 256 threads with 4 x 4 register tiles (mm_nt), x and omega rows
// of the whole width D in shared memory.
template <typename T, int D>
__global__ void __launch_bounds__(256) simt_project(const T *__restrict__ x, const float *__restrict__ omega,
                                                    float *__restrict__ P, int H, int L, int nproj, int identity) {
    constexpr int TT = 64, NT = 64, DP = D + 4;
    extern __shared__ float4 sm4[];
    float *xs = reinterpret_cast<float *>(sm4);   // [TT][DP]
    float *ws = xs + TT * DP;                     // [NT][DP]
    const int bh = blockIdx.z, h = bh % H;
    const int t0 = blockIdx.x * TT, n0 = blockIdx.y * NT;
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const T *xb = x + (size_t)bh * L * D;
    // 4 values per load (rows of D values: D % 4 == 0)
#pragma unroll
    for (int e = tid; e < TT * D / 4; e += 256) {
        const int t = e / (D / 4), j = 4 * (e % (D / 4));
        *reinterpret_cast<float4 *>(xs + t * DP + j) =
            t0 + t < L ? load4_in(xb, (size_t)(t0 + t) * D + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int e = tid; e < NT * D / 4; e += 256) {
        const int n = e / (D / 4), j = 4 * (e % (D / 4));
        float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
        if (n0 + n < nproj) {
            if (identity) {
                const int c = n0 + n - j;   // the 1 of row n0 + n, if among columns j .. j + 3
                w = make_float4(c == 0, c == 1, c == 2, c == 3);
            } else {
                w = *reinterpret_cast<const float4 *>(omega + ((size_t)h * nproj + n0 + n) * D + j);
            }
        }
        *reinterpret_cast<float4 *>(ws + n * DP + j) = w;
    }
    __syncthreads();
    float acc[4][4] = {};
    mm_nt(acc, xs, DP, ws, DP, D, ty, tx);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int t = t0 + ty + 16 * u;
        if (t >= L) continue;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const int n = n0 + tx + 16 * w;
            if (n < nproj) P[((size_t)bh * L + t) * nproj + n] = acc[u][w];
        }
    }
}

template <typename T, int D>
int project_launch(const T *x, const float *omega, float *P, const Problem &p, cudaStream_t st) {
    const size_t smem = sizeof(float) * 2 * 64 * (D + 4);
    if (cudaFuncSetAttribute(simt_project<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess) {
        cudaGetLastError();
        return FAVOR_ERR_CUDA;
    }
    const dim3 pg((p.L + 63) / 64, (p.nproj + 63) / 64, p.BH);
    simt_project<T, D><<<pg, 256, smem, st>>>(x, omega, P, p.H, p.L, p.nproj, map_is_elementwise(p.map));
    return FAVOR_OK;
}

// 2. features: one warp per token row.
template <typename T>
__global__ void simt_features(const T *__restrict__ x, const float *__restrict__ P,
                              float *__restrict__ phi, float *__restrict__ logscale, int BH,
                              int L, int d, int m, int nproj, int r, int map) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= BH * L) return;
    const size_t row = (size_t)warp;
    const float *pr = P + row * nproj;
    float *fr = phi + row * r;
    if (map_is_elementwise(map)) {
        for (int n = lane; n < nproj; n += 32) {
            float t = pr[n];
            fr[n] = map == FAVOR_MAP_RELU ? fmaxf(t, 0.f) : (t > 0.f ? t + 1.f : expf(t));
        }
        if (lane == 0) logscale[row] = 0.f;
        return;
    }
    if (map_is_trig(map)) {
        for (int n = lane; n < nproj; n += 32) {
            float s, c;
            sincosf(pr[n], &s, &c);
            fr[2 * n] = s;
            fr[2 * n + 1] = c;
        }
        // the softmax-scaled map: exp(|x|^2/2) in the row's log-scale
        float nrm = 0.f;
        if (map == FAVOR_MAP_TRIG_SOFTMAX) {
            const T *xr = x + row * d;
            for (int j = lane; j < d; j += 32) {
                float t = load_in(xr, j);
                nrm = fmaf(t, t, nrm);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) nrm += __shfl_xor_sync(0xffffffffu, nrm, o);
        }
        if (lane == 0) logscale[row] = 0.5f * nrm - 0.5f * logf((float)m);
        return;
    }
    float mx = -INFINITY;
    for (int n = lane; n < nproj; n += 32) mx = fmaxf(mx, pr[n]);
    float nrm = 0.f;
    const T *xr = x + row * d;
    for (int j = lane; j < d; j += 32) {
        float t = load_in(xr, j);
        nrm = fmaf(t, t, nrm);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        nrm += __shfl_xor_sync(0xffffffffu, nrm, o);
    }
    for (int n = lane; n < nproj; n += 32) fr[n] = expf(pr[n] - mx);
    if (lane == 0) logscale[row] = mx - 0.5f * nrm - 0.5f * logf((float)m);
}

// 3a. per-head maximum of the key log-scales.
__global__ void simt_head_max(const float *__restrict__ logscale, float *__restrict__ hmax, int L) {
    __shared__ float red[32];
    const int bh = blockIdx.x;
    float mx = -INFINITY;
    for (int t = threadIdx.x; t < L; t += blockDim.x) mx = fmaxf(mx, logscale[(size_t)bh * L + t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x < 32) {
        int nw = blockDim.x >> 5;
        mx = threadIdx.x < nw ? red[threadIdx.x] : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (threadIdx.x == 0) hmax[bh] = mx;
    }
}

// 3b. phi_K <- phi~_K * exp(logscale - head max)
// (a warp per row: the row's factor once, 16 bytes at a time; r % 4 == 0)
__global__ void simt_key_scale(float *__restrict__ phi, const float *__restrict__ logscale,
                               const float *__restrict__ hmax, int L, int r, size_t rows) {
    const int lane = threadIdx.x & 31;
    const size_t nwarp = (size_t)gridDim.x * blockDim.x / 32;
    for (size_t row = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) / 32; row < rows; row += nwarp) {
        const float sc = expf(logscale[row] - hmax[row / L]);
        float4 *p4 = reinterpret_cast<float4 *>(phi + row * r);
        for (int c = lane; c < r / 4; c += 32) {
            float4 x = p4[c];
            x.x *= sc;
            x.y *= sc;
            x.z *= sc;
            x.w *= sc;
            p4[c] = x;
        }
    }
}

// The state of a run of keys (the decode state of a prefix, [r][dv + 1]):
// dS[f][c] = sum_{t in [t0, t1)} phi_K[t][f] * (c < dv ? v[t][c] : 1);
// grid (ceil(r/32), dv+1, BH*nseg); segment length seg.
template <typename T>
__global__ void simt_state(const float *__restrict__ phik, const T *__restrict__ v,
                           float *__restrict__ S, int L, int r, int dv, int seg, int nseg) {
    const int f = blockIdx.x * 32 + threadIdx.x;
    const int c = blockIdx.y;
    const int bh = blockIdx.z / nseg, s = blockIdx.z % nseg;
    if (f >= r) return;
    const int t0 = s * seg, t1 = min(L, t0 + seg);
    const float *pk = phik + (size_t)bh * L * r;
    const T *vb = v + (size_t)bh * L * dv;
    float acc = 0.f;
    for (int t = t0; t < t1; ++t) {
        float vv = c < dv ? load_in(vb, (size_t)t * dv + c) : 1.f;
        acc = fmaf(pk[(size_t)t * r + f], vv, acc);
    }
    S[(((size_t)bh * nseg + s) * r + f) * (dv + 1) + c] = acc;
}
template <typename T>
int features_into(const T *x, const float *omega, float *P, float *phi, float *logscale,
                  const Problem &p, cudaStream_t st) {
    const int prc = p.d == 32   ? project_launch<T, 32>(x, omega, P, p, st)
                    : p.d == 64 ? project_launch<T, 64>(x, omega, P, p, st)
                                : project_launch<T, 128>(x, omega, P, p, st);
    if (prc != FAVOR_OK) return prc;
    FAVOR_LAUNCH_CHECK();
    long long rows = (long long)p.BH * p.L;
    simt_features<T><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, st>>>(
        x, P, phi, logscale, p.BH, p.L, p.d, p.m, p.nproj, p.r, p.map);
    FAVOR_LAUNCH_CHECK();
    return FAVOR_OK;
}

}  // namespace


namespace {
template <typename T>
int key_state_t(const T *k, const T *v, const float *omega, const Problem &p, cudaStream_t st,
                const float **S_out, const float **hmax_out) {
    const size_t rows = (size_t)p.BH * p.L;
    const size_t per = (size_t)p.r * (p.dv + 1);
    size_t bytes = carve_bytes<float>(rows * p.nproj) + carve_bytes<float>(rows * p.r) +
                   carve_bytes<float>(rows) + carve_bytes<float>(p.BH) + carve_bytes<float>((size_t)p.BH * per);
    int status = FAVOR_OK;
    void *ws = workspace(bytes, &status);
    if (!ws) return status;
    Carve cv{static_cast<char *>(ws), 0};
    float *P = cv.take<float>(rows * p.nproj);
    float *phik = cv.take<float>(rows * p.r);
    float *lsk = cv.take<float>(rows);
    float *hmax = cv.take<float>(p.BH);
    float *S = cv.take<float>((size_t)p.BH * per);
    int rc = features_into<T>(k, omega, P, phik, lsk, p, st);
    if (rc) return rc;
    simt_head_max<<<p.BH, 256, 0, st>>>(lsk, hmax, p.L);
    FAVOR_LAUNCH_CHECK();
    const unsigned sg = (unsigned)std::min<size_t>((rows * 32 + 255) / 256, 152 * 64);
    simt_key_scale<<<sg, 256, 0, st>>>(phik, lsk, hmax, p.L, p.r, rows);
    FAVOR_LAUNCH_CHECK();
    dim3 sgrid((p.r + 31) / 32, p.dv + 1, p.BH);
    simt_state<T><<<sgrid, 32, 0, st>>>(phik, v, S, p.L, p.r, p.dv, p.L, 1);
    FAVOR_LAUNCH_CHECK();
    *S_out = S;
    *hmax_out = hmax;
    return FAVOR_OK;
}
}  // namespace

int simt_key_state(const void *k, const void *v, bool bf16_in, const float *omega, const Problem &p,
                   cudaStream_t st, const float **S, const float **hmax) {
    if (bf16_in)
        return key_state_t<uint16_t>(static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(v),
                                     omega, p, st, S, hmax);
    return key_state_t<float>(static_cast<const float *>(k), static_cast<const float *>(v), omega, p, st,
                              S, hmax);
}

int simt_feature_map(const void *x, bool bf16_in, const float *omega, float *phi,
                     float *log_scale, const Problem &p, cudaStream_t stream) {
    const size_t rows = (size_t)p.BH * p.L;
    int status = FAVOR_OK;
    float *P = static_cast<float *>(workspace(carve_bytes<float>(rows * p.nproj), &status));
    if (!P) return status;
    if (bf16_in)
        return features_into<uint16_t>(static_cast<const uint16_t *>(x), omega, P, phi, log_scale,
                                       p, stream);
    return features_into<float>(static_cast<const float *>(x), omega, P, phi, log_scale, p, stream);
}

// ---------------------------------------------------------------------------
// Backward pass (fp32 SIMT): the gradients of a loss given g = dloss/dout,
//   dnum_i = g_i / den_i,  dden_i = -(g_i . out_i) / den_i
//   dphi(q_i) = S_i dnum_i + z_i dden_i
//   dphi(k_j) = R_j v_j + rho_j,  dv_j = R_j^T phi(k_j),
//   R_j = sum_{i >= j} phi(q_i) dnum_i^T,  rho_j = sum_{i >= j} phi(q_i) dden_i
// (non-causal: S, z, R, rho over all rows), then the feature maps'
// derivatives to dq, dk and dw -- the prefix sums of the Performer study
// notes ("Case 2") accumulated in reverse.  In chunks of 64 rows: the states
// entering (S) and leaving (R) a chunk plus the masked products inside it,
//   A_ij = phi(q_i).phi(k_j),  B_ij = dnum_i.v_j + dden_i   (j <= i).
// The stabilised features of the forward pass serve as the features (out
// does not change under them); the map derivatives use the products
// dphi_f phi_f (positive map) or the scale applied to the raw sin, cos (trig
// maps), which are the same for the stabilised and the exact features.
// ---------------------------------------------------------------------------
namespace {

constexpr int kBwdRows = 64;    // rows per chunk of the SIMT forward and backward passes
constexpr int kBwdThreads = 256;   // threads of a bwd_chunk block

// dphi_q, dphi_k [rows][r] and dv [rows][dv] of a chunk of C = 64 rows from the
// entering state S, the leaving state R and (causal) the masked A, B inside
// it; block per (chunk, head), 256 threads, 64-feature tiles (two blocks per
// SM at dv = 64):
//   B = Y [V | 1]^T, masked to j <= i
//   pass 1: dv += phi_k R[:, :dv]; then dv += A^T dnum (A masked, from chunk_rows)
//   pass 2: dphi_q = Y S^T + B phi_k, then dphi_k = [V | 1] R^T + B^T phi_q
// A thread owns rows 4 ty .. 4 ty + 3, so the triangular products (B phi_k,
// B^T phi_q, A^T dnum) run only over the keys or queries on its side of the
// diagonal.
template <typename T, int DV>
__global__ void __launch_bounds__(kBwdThreads, DV <= 64 ? 2 : 1) bwd_chunk(const float *__restrict__ phiq, const float *__restrict__ phik,
                                                 const T *__restrict__ v, const float *__restrict__ Sin,
                                                 const float *__restrict__ Rout, const float *__restrict__ Y,
                                                 const float *__restrict__ Am, float *__restrict__ dphiq,
                                                 float *__restrict__ dphik, float *__restrict__ dV, int L, int r,
                                                 int nst, int causal) {
    constexpr int C = kBwdRows, FT = 64, P = FT + 4, W = DV + 1, WP = DV + 4, NG = (DV + 63) / 64;
    constexpr int NT = kBwdThreads;
    static_assert(NT == 256, "the tiled products assume 256 threads");
    extern __shared__ float4 sm4[];
    float *Ys = reinterpret_cast<float *>(sm4);   // [C][WP]  dnum | dden | 0
    float *Vs = Ys + C * WP;                      // [C][WP]  v | 1 | 0
    float *Bs = Vs + C * WP;                      // [C][P]   B
    float *X1 = Bs + C * P;                       // [C][P]   phi_q (pass 1), A (after it), phi_k (pass 2)
    float *X2 = X1 + C * P;                       // [C][P]   phi_k (pass 1), phi_q (pass 2)
    float *Ts = X2 + C * P;                       // R tile [FT][WP] (pass 1); S^T, R^T [WP][P] (pass 2)
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const int ch = blockIdx.x, bh = blockIdx.y, t0 = ch * C, n = min(C, L - t0);
    const size_t row0 = (size_t)bh * L + t0;
    const size_t st = ((size_t)bh * nst + (causal ? ch : 0)) * r * WP;
    const float *S = Sin + st, *R = Rout + st;
#pragma unroll 4
    for (int e = tid; e < C * WP / 4; e += NT) {   // Y rows have the same pitch (zero pad columns)
        const int i = e / (WP / 4), c = 4 * (e % (WP / 4));
        *reinterpret_cast<float4 *>(Ys + 4 * e) =
            i < n ? *reinterpret_cast<const float4 *>(Y + (row0 + i) * WP + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll 4
    for (int e = tid; e < C * WP; e += NT) {
        const int i = e / WP, c = e % WP;
        Vs[e] = (i < n && c < W) ? (c < DV ? load_in(v, (row0 + i) * DV + c) : 1.f) : 0.f;
    }
    // rows x 64 features of phi (phiq or phik) into a [C][P] tile
    auto load_x = [&](float *dst, const float *src, int f0) {
        float4 t[C * FT / 4 / NT];
#pragma unroll
        for (int k = 0; k < C * FT / 4 / NT; ++k) {
            const int e = tid + NT * k, i = e / (FT / 4), f = 4 * (e % (FT / 4));
            t[k] = (i < n && f0 + f < r) ? *reinterpret_cast<const float4 *>(src + (row0 + i) * r + f0 + f)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);   // r % 4 == 0
        }
#pragma unroll
        for (int k = 0; k < C * FT / 4 / NT; ++k) {
            const int e = tid + NT * k, i = e / (FT / 4), f = 4 * (e % (FT / 4));
            *reinterpret_cast<float4 *>(dst + i * P + f) = t[k];
        }
    };
    // state rows f0 .. f0 + 63 (pitch WP, 16 bytes at a time) transposed into [WP][P]
    constexpr int NS = (FT * WP / 4 + NT - 1) / NT;
    auto fetch_st = [&](const float *src, int f0, float4(&t)[NS]) {
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const int e = tid + NT * k, f = e / (WP / 4), c = 4 * (e % (WP / 4));
            t[k] = (e < FT * WP / 4 && f0 + f < r) ? *reinterpret_cast<const float4 *>(src + (size_t)(f0 + f) * WP + c)
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    auto load_st = [&](const float *src, int f0) {
        float4 t[NS];
        fetch_st(src, f0, t);
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const int e = tid + NT * k, f = e / (WP / 4), c = 4 * (e % (WP / 4));
            if (e < FT * WP / 4) {
                Ts[(c + 0) * P + f] = t[k].x;
                Ts[(c + 1) * P + f] = t[k].y;
                Ts[(c + 2) * P + f] = t[k].z;
                Ts[(c + 3) * P + f] = t[k].w;
            }
        }
    };
    __syncthreads();
    if (causal) {
        float b[4][4] = {};
        mm_nt<4, 16, true>(b, Ys, WP, Vs, WP, WP, ty, tx);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int i = 4 * ty + u, j = tx + 16 * w;
                Bs[i * P + j] = j <= i ? b[u][w] : 0.f;
            }
    }
    // ---- pass 1 (R tile row-major [f][WP]; its pad columns are never read)
    float dvr[NG][4][4] = {};
    for (int f0 = 0; f0 < r; f0 += FT) {
        __syncthreads();
        load_x(X2, phik, f0);
        {
            float4 t[NS];
            fetch_st(R, f0, t);
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const int e = tid + NT * k;
                if (e < FT * WP / 4) *reinterpret_cast<float4 *>(Ts + 4 * e) = t[k];   // [FT][WP], same pitch
            }
        }
        __syncthreads();
#pragma unroll
        for (int g = 0; g < NG; ++g)
            if (64 * g + 4 * tx < DV) mm_nn<4, 16, true>(dvr[g], X2, P, Ts + 64 * g, WP, FT, ty, tx);
    }
    __syncthreads();
    if (causal) {   // the masked A of this chunk, row-major
        const float *src = Am + ((size_t)bh * nst + ch) * C * C;
#pragma unroll
        for (int k = 0; k < C * C / 4 / NT; ++k) {
            const int e = tid + NT * k, i = e / (C / 4), j = 4 * (e % (C / 4));
            *reinterpret_cast<float4 *>(X1 + i * P + j) = *reinterpret_cast<const float4 *>(src + i * C + j);
        }
    }
    // pad rows W .. WP - 1 of the transposed state tiles stay zero through pass 2
    for (int e = tid; e < (WP - W) * P; e += NT) Ts[W * P + e] = 0.f;
    __syncthreads();
    if (causal) {
#pragma unroll
        for (int g = 0; g < NG; ++g)
            if (64 * g + 4 * tx < DV) mm_tn<true>(dvr[g], X1, P, Ys + 64 * g, WP, C, ty, tx, 4 * ty);   // i >= j
    }
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = 4 * ty + u, c = 64 * g + 4 * tx;
            if (j < n && c < DV)
                *reinterpret_cast<float4 *>(dV + (row0 + j) * DV + c) =
                    make_float4(dvr[g][u][0], dvr[g][u][1], dvr[g][u][2], dvr[g][u][3]);
        }
    // ---- pass 2
    for (int f0 = 0; f0 < r; f0 += FT) {
        __syncthreads();
        load_x(X1, phik, f0);
        load_x(X2, phiq, f0);
        load_st(S, f0);
        __syncthreads();
        {
            float dq[4][4] = {};
            mm_nn<4, 16, true>(dq, Ys, WP, Ts, P, WP, ty, tx);
            if (causal) mm_nn<4, 16, true>(dq, Bs, P, X1, P, 4 * ty + 4, ty, tx);   // j <= i
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = 4 * ty + u, f = f0 + 4 * tx;
                if (i < n && f < r)
                    *reinterpret_cast<float4 *>(dphiq + (row0 + i) * r + f) =
                        make_float4(dq[u][0], dq[u][1], dq[u][2], dq[u][3]);
            }
        }
        __syncthreads();
        load_st(R, f0);
        __syncthreads();
        {
            float dk[4][4] = {};
            mm_nn<4, 16, true>(dk, Vs, WP, Ts, P, WP, ty, tx);
            if (causal) mm_tn<true>(dk, Bs, P, X2, P, C, ty, tx, 4 * ty);   // j >= i
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = 4 * ty + u, f = f0 + 4 * tx;
                if (i < n && f < r)
                    *reinterpret_cast<float4 *>(dphik + (row0 + i) * r + f) =
                        make_float4(dk[u][0], dk[u][1], dk[u][2], dk[u][3]);
            }
        }
    }
}

template <typename T, int DV>
constexpr size_t bwd_chunk_smem() {
    return sizeof(float) * (2 * kBwdRows * (DV + 4) + 3 * kBwdRows * 68 +
                            ((DV + 4) * 68 > 64 * (DV + 4) ? (DV + 4) * 68 : 64 * (DV + 4)));
}

// per (row, projection p): the coefficient c of the map derivative, in place
// of the projection P[row][p]:
//   positive: c = dphi_p phi_p              (dx = sum_p c w_p - x sum_p c)
//   trig:     c = s (dphi_2p cos P - dphi_2p+1 sin P), s the scale on the raw
//             sin, cos of that row           (dx = sum_p c w_p [+ x tot])
//   elu1, relu: c = dphi_p phi'(x_p)        (dx = c)
__global__ void bwd_coeff(float *__restrict__ P, const float *__restrict__ dphi, const float *__restrict__ phi,
                          const float *__restrict__ logscale, const float *__restrict__ hmax, size_t rows, int L,
                          int nproj, int r, int map, int is_key) {
    const size_t total = rows * nproj;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
        const size_t row = e / nproj;
        const int p = (int)(e % nproj);
        const float a = P[e];
        float c;
        if (map == FAVOR_MAP_POSITIVE) {
            c = dphi[row * r + p] * phi[row * r + p];
        } else if (map_is_trig(map)) {
            // keys carry exp(logscale - head max) on the raw sin, cos; queries 1
            const float s = is_key ? expf(logscale[row] - hmax[row / L]) : 1.f;
            float sn, cs;
            sincosf(a, &sn, &cs);
            c = s * (dphi[row * r + 2 * p] * cs - dphi[row * r + 2 * p + 1] * sn);
        } else {
            const float der = a > 0.f ? 1.f : (map == FAVOR_MAP_ELU1 ? expf(a) : 0.f);
            c = dphi[row * r + p] * der;
        }
        P[e] = c;
    }
}

// dx [rows][d] from the coefficients, 64 rows of one head per block (256
// threads): dx = C w_h (C [rows][nproj] and w_h [nproj][d] in 64-projection
// tiles, register-tiled, read a tile ahead into registers), then the map's row
// term: positive - x sum_p C[p]; softmax-scaled trig + x sum_f dphi_f phi_f;
// elementwise maps dx = C.  For the positive map the coefficients
// C = dphi phi are formed here from the feature gradients and written to C
// (the omega gradient reads them); the other maps take C from bwd_coeff.
// Thread (ty, tx) owns rows ty + 16 u and columns 4 tx + w (+ 64 per group).
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_dx(float *__restrict__ C, const float *__restrict__ dphi,
                                              const float *__restrict__ phi, const T *__restrict__ x,
                                              const float *__restrict__ omega, float *__restrict__ dx, int L, int H,
                                              int nproj, int r, int map) {
    constexpr int RB = 64, PT = 64, P = PT + 4, DP = D + 4, NG = (D + 63) / 64, NT = 256;
    constexpr int NX = RB * PT / 4 / NT, NW = (PT * D / 4 + NT - 1) / NT;
    extern __shared__ float4 sm4[];
    float *Cs = reinterpret_cast<float *>(sm4);   // [RB][P]  coefficients
    float *Ws = Cs + RB * P;                      // [PT][DP] projections w_p
    float *tot = Ws + PT * DP;                    // [RB]     row term (softmax-scaled trig)
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const int t0 = blockIdx.x * RB, bh = blockIdx.y, h = bh % H, n = min(RB, L - t0);
    const size_t row0 = (size_t)bh * L + t0;
    if (map_is_elementwise(map)) {
        for (int e = tid; e < n * D; e += NT) dx[row0 * D + e] = C[row0 * nproj + e];
        return;
    }
    const bool pos = map == FAVOR_MAP_POSITIVE;
    if (map == FAVOR_MAP_TRIG_SOFTMAX) {
        const int warp = tid >> 5, lane = tid & 31;
        for (int i = warp; i < RB; i += NT / 32) {
            float sv = 0.f;
            if (i < n)
                for (int f = lane; f < r; f += 32) sv = fmaf(dphi[(row0 + i) * r + f], phi[(row0 + i) * r + f], sv);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, o);
            if (lane == 0) tot[i] = sv;
        }
    }
    const float *w = omega + (size_t)h * nproj * D;
    // staged a tile ahead: the coefficients (other maps) or dphi and phi
    // (positive map, multiplied when the tile is put in shared memory)
    float4 xc[NX], xf[NX], xw[NW];
    auto fetch = [&](int p0) {
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NX; ++k) {
            const int e = tid + NT * k, i = e / (PT / 4), pp = 4 * (e % (PT / 4));
            xc[k] = xf[k] = z;
            if (i < n && p0 + pp < nproj) {   // nproj % 4 == 0
                const size_t o = (row0 + i) * nproj + p0 + pp;
                if (pos) {   // positive map: r == nproj
                    xc[k] = *reinterpret_cast<const float4 *>(dphi + o);
                    xf[k] = *reinterpret_cast<const float4 *>(phi + o);
                } else {
                    xc[k] = *reinterpret_cast<const float4 *>(C + o);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const int e = tid + NT * k, pp = e / (D / 4), j = 4 * (e % (D / 4));
            xw[k] = (e < PT * D / 4 && p0 + pp < nproj) ? *reinterpret_cast<const float4 *>(w + (size_t)(p0 + pp) * D + j)
                                                       : z;
        }
    };
    float acc[NG][4][4] = {}, rs[4] = {};
    fetch(0);
    for (int p0 = 0; p0 < nproj; p0 += PT) {
        __syncthreads();
#pragma unroll
        for (int k = 0; k < NX; ++k) {
            const int e = tid + NT * k, i = e / (PT / 4), pp = 4 * (e % (PT / 4));
            float4 cv = xc[k];
            if (pos) {
                cv = make_float4(cv.x * xf[k].x, cv.y * xf[k].y, cv.z * xf[k].z, cv.w * xf[k].w);
                if (i < n && p0 + pp < nproj)
                    *reinterpret_cast<float4 *>(C + (row0 + i) * nproj + p0 + pp) = cv;   // for the omega gradient
            }
            *reinterpret_cast<float4 *>(Cs + i * P + pp) = cv;
        }
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const int e = tid + NT * k, pp = e / (D / 4), j = 4 * (e % (D / 4));
            if (e < PT * D / 4) *reinterpret_cast<float4 *>(Ws + pp * DP + j) = xw[k];
        }
        __syncthreads();
        if (p0 + PT < nproj) fetch(p0 + PT);
        if (pos) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 cv = *reinterpret_cast<const float4 *>(Cs + (ty + 16 * u) * P + 4 * tx);
                rs[u] += (cv.x + cv.y) + (cv.z + cv.w);
            }
        }
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
            if (64 * gi + 4 * tx < D) mm_nn(acc[gi], Cs, P, Ws + 64 * gi, DP, PT, ty, tx);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) rs[u] += __shfl_xor_sync(0xffffffffu, rs[u], o);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = ty + 16 * u;
        if (i >= n) continue;
        const float term = pos ? -rs[u] : (map == FAVOR_MAP_TRIG_SOFTMAX ? tot[i] : 0.f);
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            const int j = 64 * gi + 4 * tx;
            if (j >= D) continue;
            const size_t o = (row0 + i) * D + j;
            const float4 xv = load4_in(x, o);
            *reinterpret_cast<float4 *>(dx + o) =
                make_float4(fmaf(term, xv.x, acc[gi][u][0]), fmaf(term, xv.y, acc[gi][u][1]),
                            fmaf(term, xv.z, acc[gi][u][2]), fmaf(term, xv.w, acc[gi][u][3]));
        }
    }
}

// The chunk states of a head in one pass over its chunks: the state of chunk c
// is St_c[f][col] = sum_{rows of c} phi[row][f] Yc[row][col], col <= dv, with
// Yc = [v | 1] (forward) or the rows' [dnum | dden] (backward).  Written per
// chunk: causal, the exclusive prefix (forward: chunks before c; reverse:
// chunks after c); non-causal, the total of the z-th of gridDim.z ranges of
// chunks into slot z (state_sum adds them).  S holds nslot slots per head.
// Causal with gridDim.z > 1 (the forward pass with few heads): each range of
// chunks starts from zero and writes its total into tot [BH][ranges][r][dv + 4];
// range_offsets turns the totals into each range's offset, which chunk_rows
// adds to the states it reads.
// Block per (64-feature tile, head, range), 256 threads, the chunks in order
// (a fixed summation order), the next chunk's rows read into registers while
// the current one is added; thread (ty, tx) owns features 4 ty + u and columns
// 4 tx + w (+ 64 per group) of the running state, and every thread the last
// column (sum of phi, or of phi dden) of its features.
// The instance that reads v at dv = 128 loads each chunk straight into shared
// memory instead: without the staged chunk it fits 128 registers, two blocks
// per SM, and the forward pass gives it twice the chunk ranges.
template <int DV, bool YIN>
__host__ __device__ constexpr bool state_scan_staged() {
    return YIN || DV <= 64;
}

template <typename T, int DV, bool YIN>
__global__ void __launch_bounds__(256, (DV <= 64 || !state_scan_staged<DV, YIN>()) ? 2 : 1) state_scan(const float *__restrict__ phi, const T *__restrict__ v,
                                                     const float *__restrict__ Y, float *__restrict__ S,
                                                     float *__restrict__ tot, int L, int r, int nch, int nslot,
                                                     int causal, int reverse) {
    constexpr int C = kBwdRows, FT = 64, P = FT + 4, WP = DV + 4, NG = (DV + 63) / 64, NT = 256;
    constexpr int NX = C * FT / 4 / NT;
    extern __shared__ float4 sm4[];
    float *Ps = reinterpret_cast<float *>(sm4);   // [C][P]  phi rows x this block's 64 features
    float *Ys = Ps + C * P;                       // [C][WP] Yc | 0
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const int f0 = blockIdx.x * FT, bh = blockIdx.y;
    constexpr int NY4 = (C * WP / 4 + NT - 1) / NT, NV4 = (C * DV / 4 + NT - 1) / NT;
    constexpr bool STAGED = state_scan_staged<DV, YIN>();
    // the 16-byte pieces of chunk ch that thread tid moves: phi rows (k < NX), v rows (k < NV4)
    auto p4 = [&](int k, int ch) {
        const int t0 = ch * C, n = min(C, L - t0), e = tid + NT * k, i = e / (FT / 4), f = 4 * (e % (FT / 4));
        return (i < n && f0 + f < r) ? *reinterpret_cast<const float4 *>(phi + ((size_t)bh * L + t0 + i) * r + f0 + f)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);   // r % 4 == 0
    };
    auto v4 = [&](int k, int ch) {
        const int t0 = ch * C, n = min(C, L - t0), e = tid + NT * k, i = e / (DV / 4), c = 4 * (e % (DV / 4));
        return (e < C * DV / 4 && i < n) ? load4_raw(v, ((size_t)bh * L + t0 + i) * DV + c) : make_uint4(0u, 0u, 0u, 0u);
    };
    float4 xp[STAGED ? NX : 1], xy4[YIN ? NY4 : 1];   // Y rows (pitch WP), 16 bytes at a time
    uint4 xv[(YIN || !STAGED) ? 1 : NV4];             // v rows, 4 values a load (bits, converted when put)
    int nstaged = 0;                                  // valid rows of the staged chunk
    auto fetch = [&](int ch) {
        const int t0 = ch * C, n = min(C, L - t0);
        const size_t row0 = (size_t)bh * L + t0;
#pragma unroll
        for (int k = 0; k < NX; ++k) xp[k] = p4(k, ch);
        if constexpr (YIN) {
#pragma unroll
            for (int k = 0; k < NY4; ++k) {
                const int e = tid + NT * k, i = e / (WP / 4), c = 4 * (e % (WP / 4));
                xy4[k] = (e < C * WP / 4 && i < n) ? *reinterpret_cast<const float4 *>(Y + (row0 + i) * WP + c)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        } else {
#pragma unroll
            for (int k = 0; k < NV4; ++k) xv[k] = v4(k, ch);
            nstaged = n;
        }
    };
    for (int e = tid; e < C * WP; e += NT) Ys[e] = 0.f;   // pad columns stay zero
    float acc[NG][4][4] = {}, zc[4] = {};   // zc: the last column (every tx holds it)
    auto write_state = [&](float *dst) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float z = zc[u];
            const int f = f0 + 4 * ty + u;
            if (f >= r) continue;
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
                const int c = 64 * gi + 4 * tx;
                if (c < DV)
                    *reinterpret_cast<float4 *>(dst + (size_t)f * WP + c) =
                        make_float4(acc[gi][u][0], acc[gi][u][1], acc[gi][u][2], acc[gi][u][3]);
            }
            if (tx == 0) *reinterpret_cast<float4 *>(dst + (size_t)f * WP + DV) = make_float4(z, 0.f, 0.f, 0.f);
        }
    };
    // this block's chunks: all (causal) or the z-th range (non-causal)
    const int per_z = (nch + gridDim.z - 1) / gridDim.z, c_lo = blockIdx.z * per_z, c_n = min(nch, c_lo + per_z) - c_lo;
    if constexpr (STAGED)
        if (c_n > 0) fetch(reverse ? c_lo + c_n - 1 : c_lo);
    for (int it = 0; it < c_n; ++it) {
        const int ch = reverse ? c_lo + c_n - 1 - it : c_lo + it;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < NX; ++k) {
            const int e = tid + NT * k, i = e / (FT / 4), f = 4 * (e % (FT / 4));
            *reinterpret_cast<float4 *>(Ps + i * P + f) = STAGED ? xp[k] : p4(k, ch);
        }
        if constexpr (YIN) {
#pragma unroll
            for (int k = 0; k < NY4; ++k) {
                const int e = tid + NT * k;
                if (e < C * WP / 4) *reinterpret_cast<float4 *>(Ys + 4 * e) = xy4[k];
            }
        } else {
#pragma unroll
            for (int k = 0; k < NV4; ++k) {
                const int e = tid + NT * k, i = e / (DV / 4), c = 4 * (e % (DV / 4));
                if (e < C * DV / 4) *reinterpret_cast<float4 *>(Ys + i * WP + c) = from_raw4<T>(STAGED ? xv[k] : v4(k, ch));
            }
            const int nrows = STAGED ? nstaged : min(C, L - ch * C);
            if (tid < C) Ys[tid * WP + DV] = tid < nrows ? 1.f : 0.f;   // the ones column (pads stay 0)
        }
        __syncthreads();
        if constexpr (STAGED)
            if (it + 1 < c_n) fetch(reverse ? ch - 1 : ch + 1);
        if (causal) write_state(S + ((size_t)bh * nslot + ch) * r * WP);   // exclusive: before this chunk is added
        // acc[g][u][w] += sum_i phi[i][4 ty + u] Yc[i][64 g + 4 tx + w] and the last
        // column in the same pass over the rows (one more broadcast load per row)
#pragma unroll 4
        for (int i = 0; i < C; ++i) {
            const float4 a4 = *reinterpret_cast<const float4 *>(Ps + i * P + 4 * ty);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
            const float yz = Ys[i * WP + DV];
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
                if (64 * gi + 4 * tx >= DV) continue;
                const float4 bv = *reinterpret_cast<const float4 *>(Ys + i * WP + 64 * gi + 4 * tx);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc[gi][u][0] = fmaf(av[u], bv.x, acc[gi][u][0]);
                    acc[gi][u][1] = fmaf(av[u], bv.y, acc[gi][u][1]);
                    acc[gi][u][2] = fmaf(av[u], bv.z, acc[gi][u][2]);
                    acc[gi][u][3] = fmaf(av[u], bv.w, acc[gi][u][3]);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) zc[u] = fmaf(av[u], yz, zc[u]);
        }
    }
    if (!causal) write_state(S + ((size_t)bh * nslot + blockIdx.z) * r * WP);
    else if (gridDim.z > 1) write_state(tot + ((size_t)bh * gridDim.z + blockIdx.z) * r * WP);   // the range's total
}

// causal chunk ranges: tot[bh][z] <- sum of the totals of ranges z' < z (in order)
__global__ void range_offsets(float *__restrict__ tot, int nz, size_t per, int BH) {
    const size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (e >= per * BH) return;
    float *base = tot + (e / per) * nz * per + e % per;
    float run = 0.f;
    for (int z = 0; z < nz; ++z) {
        const float t = base[(size_t)z * per];
        base[(size_t)z * per] = run;
        run += t;
    }
}

// non-causal: chunk slots 1 .. nz - 1 added to slot 0 in order
__global__ void state_sum(float *__restrict__ S, int nslot, int nz, size_t per, int BH) {
    const size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (e >= per * BH) return;
    float *base = S + (e / per) * nslot * per + e % per;
    float sum = base[0];
    for (int z = 1; z < nz; ++z) sum += base[(size_t)z * per];
    base[0] = sum;
}

// per row of a chunk: num, den from the entering state (+ the masked chunk
// sum), out = num / den; the forward pass (FWD) stores out, the backward
// pass forms dnum = g / den and dden = -(g . out) / den into
// Y [rows][dv + 4] (3 zero columns; and, causal, the masked A of the chunk
// into Am [BH][chunks][64][64] for bwd_chunk).  Block per (chunk, head), 256
// threads, 64-feature tiles read a tile ahead into registers:
//   num = phi_q S[:, :dv] (+ A_m V),  den = phi_q z (+ A_m 1),
//   A_m = (phi_q phi_k^T) masked to j <= i
// The forward instance at dv = 128 reads each tile straight into shared memory
// instead of a tile ahead into registers: without the staged tile it fits 128
// registers, so two blocks share an SM and hide each other's load latency.
template <int DV, bool FWD>
__host__ __device__ constexpr bool chunk_rows_staged() {
    return !(FWD && DV > 64);
}

template <typename T, int DV, bool FWD, typename O>
__global__ void __launch_bounds__(256, (DV <= 64 || !chunk_rows_staged<DV, FWD>()) ? 2 : 1) chunk_rows(const float *__restrict__ phiq, const float *__restrict__ phik,
                                                const T *__restrict__ v, const float *__restrict__ Sin,
                                                const float *__restrict__ g, float *__restrict__ Y,
                                                float *__restrict__ Am, O *__restrict__ out,
                                                const float *__restrict__ off, int nz, int L, int r, int nst,
                                                int causal) {
    constexpr int C = kBwdRows, FT = 64, P = FT + 4, W = DV + 1, WP = DV + 4, NG = (DV + 63) / 64, NT = 256;
    extern __shared__ float4 sm4[];
    float *Qt = reinterpret_cast<float *>(sm4);   // [C][P]   phi_q tile
    float *Kt = Qt + C * P;                       // [C][P]   phi_k tile; A_m after the feature loop
    float *Ss = Kt + C * P;                       // [FT][WP] state rows (values | z); [num | den] at the end
    float *Vs = Ss + FT * WP;                     // [C][WP]  v | 1 | 0
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const int ch = blockIdx.x, bh = blockIdx.y, t0 = ch * C, n = min(C, L - t0);
    const size_t row0 = (size_t)bh * L + t0;
    const float *S = Sin + ((size_t)bh * nst + (causal ? ch : 0)) * r * WP;
    // causal chunk ranges (forward): the offset of this chunk's range, added to its state
    const int zr = (FWD && causal && nz > 1) ? ch / ((nst + nz - 1) / nz) : 0;
    const float *O0 = zr > 0 ? off + ((size_t)bh * nz + zr) * r * WP : nullptr;
#pragma unroll 4
    for (int e = tid; e < C * WP; e += NT) {
        const int i = e / WP, c = e % WP;
        Vs[e] = (i < n && c < W) ? (c < DV ? load_in(v, (row0 + i) * DV + c) : 1.f) : 0.f;
    }
    constexpr int NX = C * FT / 4 / NT, NS = (FT * WP / 4 + NT - 1) / NT;
    constexpr bool STAGED = chunk_rows_staged<DV, FWD>();
    // the 16-byte pieces of a feature tile f0 that thread tid moves: phi_q and
    // phi_k rows (k < NX), state rows f0 .. f0 + 63 with the range offset (k < NS)
    const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
    auto q4 = [&](int k, int f0) {
        const int e = tid + NT * k, i = e / (FT / 4), f = 4 * (e % (FT / 4));
        return (i < n && f0 + f < r) ? *reinterpret_cast<const float4 *>(phiq + (row0 + i) * r + f0 + f) : zero4;
    };
    auto k4 = [&](int k, int f0) {
        const int e = tid + NT * k, i = e / (FT / 4), f = 4 * (e % (FT / 4));
        return (causal && i < n && f0 + f < r) ? *reinterpret_cast<const float4 *>(phik + (row0 + i) * r + f0 + f)
                                                : zero4;   // r % 4 == 0
    };
    auto s4 = [&](int k, int f0) {
        const int e = tid + NT * k, f = e / (WP / 4), c = 4 * (e % (WP / 4));
        if (e >= FT * WP / 4 || f0 + f >= r) return zero4;
        float4 x = *reinterpret_cast<const float4 *>(S + (size_t)(f0 + f) * WP + c);
        if (FWD && O0) {
            const float4 o = *reinterpret_cast<const float4 *>(O0 + (size_t)(f0 + f) * WP + c);
            x = make_float4(x.x + o.x, x.y + o.y, x.z + o.z, x.w + o.w);
        }
        return x;
    };
    float4 xq[STAGED ? NX : 1], xk[STAGED ? NX : 1], xs[STAGED ? NS : 1];
    auto fetch = [&](int f0) {
#pragma unroll
        for (int k = 0; k < NX; ++k) {
            xq[k] = q4(k, f0);
            xk[k] = k4(k, f0);
        }
#pragma unroll
        for (int k = 0; k < NS; ++k) xs[k] = s4(k, f0);
    };
    float a[4][4] = {}, num[NG][4][4] = {}, den[4] = {};
    if constexpr (STAGED) fetch(0);
    for (int f0 = 0; f0 < r; f0 += FT) {
        __syncthreads();
#pragma unroll
        for (int k = 0; k < NX; ++k) {
            const int e = tid + NT * k, i = e / (FT / 4), f = 4 * (e % (FT / 4));
            if constexpr (STAGED) {
                *reinterpret_cast<float4 *>(Qt + i * P + f) = xq[k];
                *reinterpret_cast<float4 *>(Kt + i * P + f) = xk[k];
            } else {
                *reinterpret_cast<float4 *>(Qt + i * P + f) = q4(k, f0);
                *reinterpret_cast<float4 *>(Kt + i * P + f) = k4(k, f0);
            }
        }
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const int e = tid + NT * k;
            if (e < FT * WP / 4)   // [FT][WP], same pitch
                *reinterpret_cast<float4 *>(Ss + 4 * e) = STAGED ? xs[k] : s4(k, f0);
        }
        __syncthreads();
        if constexpr (STAGED)
            if (f0 + FT < r) fetch(f0 + FT);
        if (causal) mm_nt(a, Qt, P, Kt, P, FT, ty, tx);
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
            if (64 * gi + 4 * tx < DV) mm_nn(num[gi], Qt, P, Ss + 64 * gi, WP, FT, ty, tx);
        // den partial over features 4 tx .. 4 tx + 3 of the tile (summed over tx below)
        const float z0 = Ss[(4 * tx) * WP + DV], z1 = Ss[(4 * tx + 1) * WP + DV], z2 = Ss[(4 * tx + 2) * WP + DV],
                    z3 = Ss[(4 * tx + 3) * WP + DV];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float4 qv = *reinterpret_cast<const float4 *>(Qt + (ty + 16 * u) * P + 4 * tx);
            den[u] = fmaf(qv.x, z0, fmaf(qv.y, z1, fmaf(qv.z, z2, fmaf(qv.w, z3, den[u]))));
        }
    }
    if (causal) {
        __syncthreads();
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int i = ty + 16 * u, j = tx + 16 * w;
                const float x = j <= i ? a[u][w] : 0.f;
                Kt[i * P + j] = x;
                if (!FWD) Am[(((size_t)bh * nst + ch) * C + i) * C + j] = x;   // for bwd_chunk
                den[u] += x;
            }
        __syncthreads();
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
            if (64 * gi + 4 * tx < DV) mm_nn(num[gi], Kt, P, Vs + 64 * gi, WP, C, ty, tx);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) den[u] += __shfl_xor_sync(0xffffffffu, den[u], o);
    // [num | den] of the chunk's rows -> shared (over the state tile), then row-wise dnum, dden
    __syncthreads();
    float *NUM = Ss;   // [C][WP]
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = ty + 16 * u;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
            if (64 * gi + 4 * tx < DV)
                *reinterpret_cast<float4 *>(NUM + i * WP + 64 * gi + 4 * tx) =
                    make_float4(num[gi][u][0], num[gi][u][1], num[gi][u][2], num[gi][u][3]);
        if (tx == 0) NUM[i * WP + DV] = den[u];
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    if constexpr (FWD) {   // the forward pass: out = num / den
        for (int e = tid; e < n * DV; e += NT) {
            const int i = e / DV, c = e % DV;
            store_out(out, (row0 + i) * DV + c, NUM[i * WP + c] / NUM[i * WP + DV]);
        }
    } else {
        for (int i = warp; i < n; i += NT / 32) {
            const float dn = NUM[i * WP + DV];
            float gdo = 0.f;
            for (int c = lane; c < DV; c += 32) {
                const float gi = g[(row0 + i) * DV + c];
                gdo = fmaf(gi, NUM[i * WP + c] / dn, gdo);
                Y[(row0 + i) * WP + c] = gi / dn;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) gdo += __shfl_xor_sync(0xffffffffu, gdo, o);
            if (lane == 0) *reinterpret_cast<float4 *>(Y + (row0 + i) * WP + DV) = make_float4(-gdo / dn, 0.f, 0.f, 0.f);
        }
    }
}

// dw[h][p][j] += over a slice of 512 of the head's rows (all batches; queries
// and keys): sum_rows c[row][p] x[row][j].  Block per (64-projection tile,
// slice, head), 256 threads, 64 rows at a time in shared memory, read a
// sub-slice ahead into registers: thread (ty, tx) owns projections 4 ty + u
// and columns 4 tx + w (+ 64 per group); one atomic add per output and block.
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_dw(const float *__restrict__ Cq, const float *__restrict__ Ck,
                                              const T *__restrict__ q, const T *__restrict__ k,
                                              float *__restrict__ dw, int B, int H, int L, int nproj) {
    constexpr int RS = 64, PT = 64, P = PT + 4, DP = D + 4, NG = (D + 63) / 64, NT = 256, SUB = 8;
    constexpr int NC = RS * PT / 4 / NT, NXD = (RS * D / 4 + NT - 1) / NT;
    extern __shared__ float4 sm4[];
    float *Cs = reinterpret_cast<float *>(sm4);   // [RS][P]  coefficient rows
    float *Xs = Cs + RS * P;                      // [RS][DP] input rows
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const int p0 = blockIdx.x * PT, h = blockIdx.z;
    float4 rc[NC];
    uint4 rx[NXD];   // input bits, converted when put in shared memory
    auto fetch = [&](int it) {   // sub-slice it / 2 of side it % 2
        const int side = it & 1, r0 = (blockIdx.y * SUB + (it >> 1)) * RS;
        const float *Cm = side ? Ck : Cq;
        const T *X = side ? k : q;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int kk = 0; kk < NC; ++kk) {
            const int e = tid + NT * kk, i = e / (PT / 4), pp = 4 * (e % (PT / 4)), t = r0 + i;
            rc[kk] = z;
            if (t < B * L && p0 + pp < nproj) {   // nproj % 4 == 0
                const size_t row = ((size_t)(t / L) * H + h) * L + t % L;
                rc[kk] = *reinterpret_cast<const float4 *>(Cm + row * nproj + p0 + pp);
            }
        }
#pragma unroll
        for (int kk = 0; kk < NXD; ++kk) {
            const int e = tid + NT * kk, i = e / (D / 4), j = 4 * (e % (D / 4)), t = r0 + i;
            rx[kk] = make_uint4(0u, 0u, 0u, 0u);
            if (e < RS * D / 4 && t < B * L) {
                const size_t row = ((size_t)(t / L) * H + h) * L + t % L;
                rx[kk] = load4_raw(X, row * D + j);
            }
        }
    };
    float acc[NG][4][4] = {};
    fetch(0);
    for (int it = 0; it < 2 * SUB; ++it) {
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < NC; ++kk) {
            const int e = tid + NT * kk, i = e / (PT / 4), pp = 4 * (e % (PT / 4));
            *reinterpret_cast<float4 *>(Cs + i * P + pp) = rc[kk];
        }
#pragma unroll
        for (int kk = 0; kk < NXD; ++kk) {
            const int e = tid + NT * kk, i = e / (D / 4), j = 4 * (e % (D / 4));
            if (e < RS * D / 4) *reinterpret_cast<float4 *>(Xs + i * DP + j) = from_raw4<T>(rx[kk]);
        }
        __syncthreads();
        if (it + 1 < 2 * SUB) fetch(it + 1);
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
            if (64 * gi + 4 * tx < D) mm_tn<true>(acc[gi], Cs, P, Xs + 64 * gi, DP, RS, ty, tx);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int p = p0 + 4 * ty + u;
        if (p >= nproj) continue;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            const int j = 64 * gi + 4 * tx;
            if (j < D) {
#pragma unroll
                for (int w = 0; w < 4; ++w) atomicAdd(&dw[((size_t)h * nproj + p) * D + j + w], acc[gi][u][w]);
            }
        }
    }
}

// dynamic shared memory of a [64][68] tile and a [64][DV + 4] tile (state_scan: DV value
// columns; bwd_dw: DV = D input columns)
template <int DV>
constexpr size_t rows64_smem() {
    return sizeof(float) * (kBwdRows * 68 + kBwdRows * (DV + 4));
}

template <int DV>
constexpr size_t chunk_rows_smem() {
    return sizeof(float) * (2 * kBwdRows * 68 + 2 * kBwdRows * (DV + 4));
}

template <typename T, int DV>
int backward_dv(const T *q, const T *k, const T *v, const float *omega, const float *g, float *dq, float *dk,
                float *dv, float *dw, const Problem &p, cudaStream_t st) {
    const size_t rows = (size_t)p.BH * p.L;
    const int nch = (p.L + kBwdRows - 1) / kBwdRows;     // chunks of 64 rows, both modes
    const size_t per = (size_t)p.r * (DV + 4);   // chunk states [r][dv + 4]: dv values, z, 3 zero columns
    size_t bytes = 2 * carve_bytes<float>(rows * p.nproj) + 4 * carve_bytes<float>(rows * p.r) +
                   2 * carve_bytes<float>(rows) + carve_bytes<float>(p.BH) +
                   2 * carve_bytes<float>((size_t)p.BH * nch * per) + carve_bytes<float>(rows * (DV + 4)) +
                   (p.causal ? carve_bytes<float>((size_t)p.BH * nch * kBwdRows * kBwdRows) : 0);
    int status = FAVOR_OK;
    void *ws = workspace(bytes, &status);
    if (!ws) return status;
    Carve cv{static_cast<char *>(ws), 0};
    float *Pq = cv.take<float>(rows * p.nproj), *Pk = cv.take<float>(rows * p.nproj);
    float *phiq = cv.take<float>(rows * p.r), *phik = cv.take<float>(rows * p.r);
    float *dphiq = cv.take<float>(rows * p.r), *dphik = cv.take<float>(rows * p.r);
    float *lsq = cv.take<float>(rows), *lsk = cv.take<float>(rows);
    float *hmax = cv.take<float>(p.BH);
    float *S = cv.take<float>((size_t)p.BH * nch * per), *R = cv.take<float>((size_t)p.BH * nch * per);
    float *Y = cv.take<float>(rows * (DV + 4));   // [rows][dv + 4]: dnum | dden | 3 zero columns
    // the masked chunk matrices A (causal), formed by chunk_rows and read by bwd_chunk
    float *Am = p.causal ? cv.take<float>((size_t)p.BH * nch * kBwdRows * kBwdRows) : nullptr;

    int rc;
    if ((rc = features_into<T>(q, omega, Pq, phiq, lsq, p, st)) || (rc = features_into<T>(k, omega, Pk, phik, lsk, p, st)))
        return rc;
    simt_head_max<<<p.BH, 256, 0, st>>>(lsk, hmax, p.L);
    FAVOR_LAUNCH_CHECK();
    const unsigned sg = (unsigned)std::min<size_t>((rows * 32 + 255) / 256, 152 * 64);
    simt_key_scale<<<sg, 256, 0, st>>>(phik, lsk, hmax, p.L, p.r, rows);
    FAVOR_LAUNCH_CHECK();
    // non-causal: the chunks in up to 8 ranges (more blocks), summed by state_sum
    const int nz = p.causal ? 1 : std::min(nch, 8);
    const dim3 cg(nch, p.BH), sg2((p.r + 63) / 64, p.BH, nz);
    const unsigned sb = (unsigned)((per * p.BH + 255) / 256);
    const size_t st_smem = rows64_smem<DV>();
    if (cudaFuncSetAttribute(state_scan<T, DV, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)st_smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(state_scan<T, DV, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)st_smem) !=
            cudaSuccess) {
        cudaGetLastError();
        return FAVOR_ERR_CUDA;
    }
    // the forward states entering each chunk (causal: exclusive prefix) or the total (chunk slot 0)
    state_scan<T, DV, false><<<sg2, 256, st_smem, st>>>(phik, v, nullptr, S, nullptr, p.L, p.r, nch, nch, p.causal, 0);
    if (nz > 1) state_sum<<<sb, 256, 0, st>>>(S, nch, nz, per, p.BH);
    FAVOR_LAUNCH_CHECK();
    {
        const size_t smem = chunk_rows_smem<DV>();
        if (cudaFuncSetAttribute(chunk_rows<T, DV, false, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess) {
            cudaGetLastError();
            return FAVOR_ERR_CUDA;
        }
        chunk_rows<T, DV, false, float><<<cg, 256, smem, st>>>(phiq, phik, v, S, g, Y, Am, nullptr, nullptr, 1,
                                                               p.L, p.r, nch, p.causal);
        FAVOR_LAUNCH_CHECK();
    }
    // the states leaving each chunk (causal: exclusive suffix) or the total
    state_scan<T, DV, true><<<sg2, 256, st_smem, st>>>(phiq, v, Y, R, nullptr, p.L, p.r, nch, nch, p.causal, 1);
    if (nz > 1) state_sum<<<sb, 256, 0, st>>>(R, nch, nz, per, p.BH);
    FAVOR_LAUNCH_CHECK();
    {
        const size_t smem = bwd_chunk_smem<T, DV>();
        if (cudaFuncSetAttribute(bwd_chunk<T, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess) {
            cudaGetLastError();
            return FAVOR_ERR_CUDA;
        }
        stats_begin(st, "bwd_chunk");
        bwd_chunk<T, DV><<<cg, kBwdThreads, smem, st>>>(phiq, phik, v, S, R, Y, Am, dphiq, dphik, dv, p.L, p.r, nch,
                                                          p.causal);
        stats_end(st);
        FAVOR_LAUNCH_CHECK();
    }
    if (p.map != FAVOR_MAP_POSITIVE) {   // the positive map's coefficients are formed in bwd_dx
        const unsigned cgr = (unsigned)std::min<size_t>((rows * p.nproj + 255) / 256, 152 * 64);
        bwd_coeff<<<cgr, 256, 0, st>>>(Pq, dphiq, phiq, lsq, hmax, rows, p.L, p.nproj, p.r, p.map, 0);
        FAVOR_LAUNCH_CHECK();
        bwd_coeff<<<cgr, 256, 0, st>>>(Pk, dphik, phik, lsk, hmax, rows, p.L, p.nproj, p.r, p.map, 1);
        FAVOR_LAUNCH_CHECK();
    }
    {
        const dim3 xg((p.L + 63) / 64, p.BH);
        auto dx_launch = [&](auto kern, int D) -> int {
            const size_t smem = sizeof(float) * (64 * 68 + 64 * (D + 4) + 64);
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
                cudaGetLastError();
                return FAVOR_ERR_CUDA;
            }
            kern<<<xg, 256, smem, st>>>(Pq, dphiq, phiq, q, omega, dq, p.L, p.H, p.nproj, p.r, p.map);
            kern<<<xg, 256, smem, st>>>(Pk, dphik, phik, k, omega, dk, p.L, p.H, p.nproj, p.r, p.map);
            return FAVOR_OK;
        };
        const int rc = p.d == 32 ? dx_launch(bwd_dx<T, 32>, 32)
                       : p.d == 64 ? dx_launch(bwd_dx<T, 64>, 64)
                                   : dx_launch(bwd_dx<T, 128>, 128);
        if (rc != FAVOR_OK) return rc;
        FAVOR_LAUNCH_CHECK();
    }
    if (dw && !map_is_elementwise(p.map)) {
        if (cudaMemsetAsync(dw, 0, (size_t)p.H * p.nproj * p.d * sizeof(float), st) != cudaSuccess) return FAVOR_ERR_CUDA;
        const dim3 wg((p.nproj + 63) / 64, (p.B * p.L + 511) / 512, p.H);
        auto dw_launch = [&](auto kern, size_t smem) -> int {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
                cudaGetLastError();
                return FAVOR_ERR_CUDA;
            }
            kern<<<wg, 256, smem, st>>>(Pq, Pk, q, k, dw, p.B, p.H, p.L, p.nproj);
            return FAVOR_OK;
        };
        // the input tile has the shape of a state tile with D columns
        const int rc = p.d == 32   ? dw_launch(bwd_dw<T, 32>, rows64_smem<32>())
                       : p.d == 64 ? dw_launch(bwd_dw<T, 64>, rows64_smem<64>())
                                   : dw_launch(bwd_dw<T, 128>, rows64_smem<128>());
        if (rc != FAVOR_OK) return rc;
        FAVOR_LAUNCH_CHECK();
    }
    return FAVOR_OK;
}

template <typename T>
int backward_t(const T *q, const T *k, const T *v, const float *omega, const float *g, float *dq, float *dk,
               float *dv, float *dw, const Problem &p, cudaStream_t st) {
    if (p.dv == 32) return backward_dv<T, 32>(q, k, v, omega, g, dq, dk, dv, dw, p, st);
    if (p.dv == 64) return backward_dv<T, 64>(q, k, v, omega, g, dq, dk, dv, dw, p, st);
    return backward_dv<T, 128>(q, k, v, omega, g, dq, dk, dv, dw, p, st);
}
// The SIMT forward pass (fp32 entry point; shapes outside the tensor-core
// layouts): features of q and k (steps 1-3), then the chunk states of the keys
// (state_scan: causal, each 64-row chunk's exclusive prefix; non-causal, the
// total) and per chunk num = phi_q S (+ A_m [V | 1]), out = num / den
// (chunk_rows in its forward mode) -- the same kernels the backward pass runs.
template <typename T, int DV>
int forward_dv(const T *q, const T *k, const T *v, const float *omega, void *out, const Problem &p,
               cudaStream_t st) {
    const size_t rows = (size_t)p.BH * p.L;
    const int nch = (p.L + kBwdRows - 1) / kBwdRows;
    // ranges of chunks per head: non-causal, up to 8 (partial totals summed by
    // state_sum); causal, enough for about one state_scan block per SM slot when the heads
    // alone give fewer (each range's offset added by chunk_rows)
    const int ntile = (p.r + 63) / 64, slots = 152 * 2;   // two state_scan blocks per SM at every dv
    const int nz = p.causal ? std::max(1, std::min(std::min(nch, 8), slots / std::max(1, ntile * p.BH)))
                            : std::min(nch, 8);
    const int nslot = p.causal ? nch : nz;
    const size_t per = (size_t)p.r * (DV + 4);
    size_t bytes = carve_bytes<float>(rows * p.nproj) + 2 * carve_bytes<float>(rows * p.r) +
                   2 * carve_bytes<float>(rows) + carve_bytes<float>(p.BH) +
                   carve_bytes<float>((size_t)p.BH * nslot * per) +
                   (p.causal && nz > 1 ? carve_bytes<float>((size_t)p.BH * nz * per) : 0);
    int status = FAVOR_OK;
    void *ws = workspace(bytes, &status);
    if (!ws) return status;
    Carve cv{static_cast<char *>(ws), 0};
    float *P = cv.take<float>(rows * p.nproj);
    float *phiq = cv.take<float>(rows * p.r), *phik = cv.take<float>(rows * p.r);
    float *lsq = cv.take<float>(rows), *lsk = cv.take<float>(rows);
    float *hmax = cv.take<float>(p.BH);
    float *S = cv.take<float>((size_t)p.BH * nslot * per);
    float *tot = p.causal && nz > 1 ? cv.take<float>((size_t)p.BH * nz * per) : nullptr;

    int rc = features_into<T>(q, omega, P, phiq, lsq, p, st);
    if (rc) return rc;
    if ((rc = features_into<T>(k, omega, P, phik, lsk, p, st))) return rc;
    simt_head_max<<<p.BH, 256, 0, st>>>(lsk, hmax, p.L);
    FAVOR_LAUNCH_CHECK();
    const unsigned sg = (unsigned)std::min<size_t>((rows * 32 + 255) / 256, 152 * 64);
    simt_key_scale<<<sg, 256, 0, st>>>(phik, lsk, hmax, p.L, p.r, rows);
    FAVOR_LAUNCH_CHECK();

    const size_t st_smem = rows64_smem<DV>(), rw_smem = chunk_rows_smem<DV>();
    if (cudaFuncSetAttribute(state_scan<T, DV, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)st_smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(chunk_rows<T, DV, true, float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)rw_smem) != cudaSuccess ||
        cudaFuncSetAttribute(chunk_rows<T, DV, true, __nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)rw_smem) != cudaSuccess) {
        cudaGetLastError();
        return FAVOR_ERR_CUDA;
    }
    state_scan<T, DV, false><<<dim3((p.r + 63) / 64, p.BH, nz), 256, st_smem, st>>>(phik, v, nullptr, S, tot, p.L,
                                                                                    p.r, nch, nslot, p.causal, 0);
    if (nz > 1) {
        const unsigned sb = (unsigned)((per * p.BH + 255) / 256);
        if (p.causal) range_offsets<<<sb, 256, 0, st>>>(tot, nz, per, p.BH);
        else state_sum<<<sb, 256, 0, st>>>(S, nslot, nz, per, p.BH);
    }
    FAVOR_LAUNCH_CHECK();
    const dim3 cg(nch, p.BH);
    stats_begin(st, "chunk_rows");
    if (p.out_bf16)
        chunk_rows<T, DV, true, __nv_bfloat16><<<cg, 256, rw_smem, st>>>(
            phiq, phik, v, S, nullptr, nullptr, nullptr, static_cast<__nv_bfloat16 *>(out), tot, nz, p.L, p.r, nslot,
            p.causal);
    else
        chunk_rows<T, DV, true, float><<<cg, 256, rw_smem, st>>>(phiq, phik, v, S, nullptr, nullptr, nullptr,
                                                                 static_cast<float *>(out), tot, nz, p.L, p.r, nslot,
                                                                 p.causal);
    stats_end(st);
    FAVOR_LAUNCH_CHECK();
    return FAVOR_OK;
}

template <typename T>
int forward_t(const T *q, const T *k, const T *v, const float *omega, void *out, const Problem &p, cudaStream_t st) {
    if (p.dv == 32) return forward_dv<T, 32>(q, k, v, omega, out, p, st);
    if (p.dv == 64) return forward_dv<T, 64>(q, k, v, omega, out, p, st);
    if (p.dv == 128) return forward_dv<T, 128>(q, k, v, omega, out, p, st);
    return FAVOR_ERR_UNSUPPORTED;
}
}  // namespace

int simt_backward(const void *q, const void *k, const void *v, bool bf16_in, const float *omega, const float *g,
                  float *dq, float *dk, float *dv, float *dw, const Problem &p, cudaStream_t stream) {
    if (bf16_in)
        return backward_t<uint16_t>(static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k),
                                    static_cast<const uint16_t *>(v), omega, g, dq, dk, dv, dw, p, stream);
    return backward_t<float>(static_cast<const float *>(q), static_cast<const float *>(k),
                             static_cast<const float *>(v), omega, g, dq, dk, dv, dw, p, stream);
}

int simt_forward(const void *q, const void *k, const void *v, bool bf16_in, const float *omega, float *out,
                 const Problem &p, cudaStream_t stream) {
    if (bf16_in)
        return forward_t<uint16_t>(static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k),
                                   static_cast<const uint16_t *>(v), omega, out, p, stream);
    return forward_t<float>(static_cast<const float *>(q), static_cast<const float *>(k), static_cast<const float *>(v),
                            omega, out, p, stream);
}

}  // namespace favor
