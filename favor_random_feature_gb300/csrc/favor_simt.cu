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
//   4b. causal       chunk states dS_c = phi_K(c)^T [V_c | 1]; exclusive prefix
//      over chunks; out_i = (phi_q S_in + sum_{j<=i in chunk} A_ij v_j) /
//      (phi_q z_in + sum_{j<=i} A_ij), A_ij = phi~_q_i . phi_K_j
//      -- study notes "Case 2" (prefix sum), diagonal included.
#include <cmath>

#include "favor_internal.h"

namespace favor {
namespace {

constexpr int kChunk = 64;   // causal chunk length of the SIMT path

__device__ __forceinline__ float load_in(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_in(const uint16_t *p, size_t i) {
    return __uint_as_float(static_cast<uint32_t>(p[i]) << 16);
}

// 1. projections: block = 32 tokens x 32 projections, x and omega tiles in smem.
template <typename T>
__global__ void simt_project(const T *__restrict__ x, const float *__restrict__ omega,
                             float *__restrict__ P, int H, int L, int d, int nproj, int identity) {
    __shared__ float xs[32][129];
    __shared__ float ws[32][129];
    const int bh = blockIdx.z, h = bh % H;
    const int t0 = blockIdx.x * 32, n0 = blockIdx.y * 32;
    const T *xb = x + (size_t)bh * L * d;
    for (int e = threadIdx.x; e < 32 * d; e += blockDim.x) {
        int t = e / d, j = e % d;
        xs[t][j] = (t0 + t < L) ? load_in(xb, (size_t)(t0 + t) * d + j) : 0.f;
    }
    for (int e = threadIdx.x; e < 32 * d; e += blockDim.x) {
        int n = e / d, j = e % d;
        float w = 0.f;
        if (n0 + n < nproj) {
            w = identity ? (n0 + n == j ? 1.f : 0.f)
                         : omega[((size_t)h * nproj + n0 + n) * d + j];
        }
        ws[n][j] = w;
    }
    __syncthreads();
    // 256 threads: thread -> (n = tid % 32, token group tid / 32 -> 4 tokens)
    const int n = threadIdx.x % 32, tg = threadIdx.x / 32;
    float acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = 0.f;
    for (int j = 0; j < d; ++j) {
        float w = ws[n][j];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = fmaf(w, xs[tg * 4 + i][j], acc[i]);
    }
    if (n0 + n < nproj) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int t = t0 + tg * 4 + i;
            if (t < L) P[((size_t)bh * L + t) * nproj + n0 + n] = acc[i];
        }
    }
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
__global__ void simt_key_scale(float *__restrict__ phi, const float *__restrict__ logscale,
                               const float *__restrict__ hmax, int L, int r, size_t total) {
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
         e += (size_t)gridDim.x * blockDim.x) {
        size_t row = e / r;
        int bh = (int)(row / L);
        phi[e] *= expf(logscale[row] - hmax[bh]);
    }
}

// 4a/4b. state reduction: dS[f][c] = sum_{t in [t0, t1)} phi_K[t][f] * (c < dv ? v[t][c] : 1)
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

// 4b. exclusive prefix over chunks, in place.
__global__ void simt_state_prefix(float *__restrict__ S, int nseg, size_t per_seg, int BH) {
    size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (e >= per_seg * BH) return;
    int bh = (int)(e / per_seg);
    size_t within = e % per_seg;
    float run = 0.f;
    for (int s = 0; s < nseg; ++s) {
        float *p = S + ((size_t)bh * nseg + s) * per_seg + within;
        float t = *p;
        *p = run;
        run += t;
    }
}

// 4a. non-causal output: thread per (row, c).
__global__ void simt_out_noncausal(const float *__restrict__ phiq, const float *__restrict__ S,
                                   float *__restrict__ out, int L, int r, int dv) {
    const int c = threadIdx.x;
    const int row = blockIdx.x * blockDim.y + threadIdx.y;
    const int bh = blockIdx.y;
    if (row >= L || c >= dv) return;
    const float *pq = phiq + ((size_t)bh * L + row) * r;
    const float *Sb = S + (size_t)bh * r * (dv + 1);
    float num = 0.f, den = 0.f;
    for (int f = 0; f < r; ++f) {
        float a = pq[f];
        num = fmaf(a, Sb[(size_t)f * (dv + 1) + c], num);
        den = fmaf(a, Sb[(size_t)f * (dv + 1) + dv], den);
    }
    out[((size_t)bh * L + row) * dv + c] = num / den;
}

// 4b. causal output: block per (chunk, head), 256 threads.
template <typename T>
__global__ void simt_out_causal(const float *__restrict__ phiq, const float *__restrict__ phik,
                                const T *__restrict__ v, const float *__restrict__ Sin,
                                float *__restrict__ out, int L, int r, int dv, int nch) {
    __shared__ float A[kChunk][kChunk + 1];
    __shared__ float den_s[kChunk];
    const int ch = blockIdx.x, bh = blockIdx.y;
    const int t0 = ch * kChunk;
    const int n = min(kChunk, L - t0);
    const float *pq = phiq + ((size_t)bh * L + t0) * r;
    const float *pk = phik + ((size_t)bh * L + t0) * r;
    const T *vb = v + ((size_t)bh * L + t0) * dv;
    const float *Sb = Sin + ((size_t)bh * nch + ch) * r * (dv + 1);
    for (int e = threadIdx.x; e < kChunk * kChunk; e += blockDim.x) {
        int i = e / kChunk, j = e % kChunk;
        float a = 0.f;
        if (i < n && j <= i) {
            for (int f = 0; f < r; ++f) a = fmaf(pq[(size_t)i * r + f], pk[(size_t)j * r + f], a);
        }
        A[i][j] = a;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        float den = 0.f;
        for (int f = 0; f < r; ++f) den = fmaf(pq[(size_t)i * r + f], Sb[(size_t)f * (dv + 1) + dv], den);
        for (int j = 0; j <= i; ++j) den += A[i][j];
        den_s[i] = den;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n * dv; e += blockDim.x) {
        int i = e / dv, c = e % dv;
        float num = 0.f;
        for (int f = 0; f < r; ++f) num = fmaf(pq[(size_t)i * r + f], Sb[(size_t)f * (dv + 1) + c], num);
        for (int j = 0; j <= i; ++j) num = fmaf(A[i][j], load_in(vb, (size_t)j * dv + c), num);
        out[((size_t)bh * L + t0 + i) * dv + c] = num / den_s[i];
    }
}

template <typename T>
int features_into(const T *x, const float *omega, float *P, float *phi, float *logscale,
                  const Problem &p, cudaStream_t st) {
    dim3 pg((p.L + 31) / 32, (p.nproj + 31) / 32, p.BH);
    simt_project<T><<<pg, 256, 0, st>>>(x, omega, P, p.H, p.L, p.d, p.nproj,
                                        map_is_elementwise(p.map));
    FAVOR_LAUNCH_CHECK();
    long long rows = (long long)p.BH * p.L;
    simt_features<T><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, st>>>(
        x, P, phi, logscale, p.BH, p.L, p.d, p.m, p.nproj, p.r, p.map);
    FAVOR_LAUNCH_CHECK();
    return FAVOR_OK;
}

template <typename T>
int forward_t(const T *q, const T *k, const T *v, const float *omega, float *out, const Problem &p,
              cudaStream_t st) {
    const size_t rows = (size_t)p.BH * p.L;
    const int nch = p.causal ? (p.L + kChunk - 1) / kChunk : 1;
    const size_t per_seg = (size_t)p.r * (p.dv + 1);
    size_t bytes = carve_bytes<float>(rows * p.nproj) + 2 * carve_bytes<float>(rows * p.r) +
                   2 * carve_bytes<float>(rows) + carve_bytes<float>(p.BH) +
                   carve_bytes<float>((size_t)p.BH * nch * per_seg);
    int status = FAVOR_OK;
    void *ws = workspace(bytes, &status);
    if (!ws) return status;
    Carve cv{static_cast<char *>(ws), 0};
    float *P = cv.take<float>(rows * p.nproj);
    float *phiq = cv.take<float>(rows * p.r);
    float *phik = cv.take<float>(rows * p.r);
    float *lsq = cv.take<float>(rows);
    float *lsk = cv.take<float>(rows);
    float *hmax = cv.take<float>(p.BH);
    float *S = cv.take<float>((size_t)p.BH * nch * per_seg);

    int rc = features_into<T>(q, omega, P, phiq, lsq, p, st);
    if (rc) return rc;
    rc = features_into<T>(k, omega, P, phik, lsk, p, st);
    if (rc) return rc;
    simt_head_max<<<p.BH, 256, 0, st>>>(lsk, hmax, p.L);
    FAVOR_LAUNCH_CHECK();
    size_t total = rows * p.r;
    unsigned sg = (unsigned)std::min<size_t>((total + 255) / 256, 152 * 64);
    simt_key_scale<<<sg, 256, 0, st>>>(phik, lsk, hmax, p.L, p.r, total);
    FAVOR_LAUNCH_CHECK();

    const int seg = p.causal ? kChunk : p.L;
    dim3 sgrid((p.r + 31) / 32, p.dv + 1, p.BH * nch);
    simt_state<T><<<sgrid, 32, 0, st>>>(phik, v, S, p.L, p.r, p.dv, seg, nch);
    FAVOR_LAUNCH_CHECK();
    if (!p.causal) {
        dim3 blk(p.dv, std::max(1, 256 / p.dv));
        dim3 og((p.L + blk.y - 1) / blk.y, p.BH);
        stats_begin(st, "simt_out_noncausal");
        simt_out_noncausal<<<og, blk, 0, st>>>(phiq, S, out, p.L, p.r, p.dv);
        stats_end(st);
        FAVOR_LAUNCH_CHECK();
        return FAVOR_OK;
    }
    size_t n = per_seg * p.BH;
    simt_state_prefix<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(S, nch, per_seg, p.BH);
    FAVOR_LAUNCH_CHECK();
    stats_begin(st, "simt_out_causal");
    simt_out_causal<T><<<dim3(nch, p.BH), 256, 0, st>>>(phiq, phik, v, S, out, p.L, p.r, p.dv, nch);
    stats_end(st);
    FAVOR_LAUNCH_CHECK();
    return FAVOR_OK;
}

}  // namespace

int simt_forward(const void *q, const void *k, const void *v, bool bf16_in, const float *omega,
                 float *out, const Problem &p, cudaStream_t stream) {
    if (bf16_in)
        return forward_t<uint16_t>(static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k),
                                   static_cast<const uint16_t *>(v), omega, out, p, stream);
    return forward_t<float>(static_cast<const float *>(q), static_cast<const float *>(k),
                            static_cast<const float *>(v), omega, out, p, stream);
}

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
    const size_t total = rows * p.r;
    const unsigned sg = (unsigned)std::min<size_t>((total + 255) / 256, 152 * 64);
    simt_key_scale<<<sg, 256, 0, st>>>(phik, lsk, hmax, p.L, p.r, total);
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

constexpr int kBwdRows = 64;    // rows per chunk (= kChunk)

// per row: out from the entering state (+ the masked chunk sum), then dnum
// and dden into Y [rows][dv + 1].  block per (chunk, head), 256 threads.
template <typename T>
__global__ void bwd_rows(const float *__restrict__ phiq, const float *__restrict__ phik, const T *__restrict__ v,
                         const float *__restrict__ Sin, const float *__restrict__ g, float *__restrict__ Y, int L,
                         int r, int dv, int nst, int causal) {
    __shared__ float A[kBwdRows][kBwdRows + 1];
    __shared__ float den_s[kBwdRows];
    const int ch = blockIdx.x, bh = blockIdx.y, t0 = ch * kBwdRows, n = min(kBwdRows, L - t0);
    const float *pq = phiq + ((size_t)bh * L + t0) * r;
    const float *pk = phik + ((size_t)bh * L + t0) * r;
    const T *vb = v + ((size_t)bh * L + t0) * dv;
    const float *S = Sin + ((size_t)bh * nst + (causal ? ch : 0)) * r * (dv + 1);
    if (causal) {
        for (int e = threadIdx.x; e < kBwdRows * kBwdRows; e += blockDim.x) {
            const int i = e / kBwdRows, j = e % kBwdRows;
            float acc = 0.f;
            if (i < n && j <= i)
                for (int f = 0; f < r; ++f) acc = fmaf(pq[(size_t)i * r + f], pk[(size_t)j * r + f], acc);
            A[i][j] = acc;
        }
        __syncthreads();
    }
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        float den = 0.f;
        for (int f = 0; f < r; ++f) den = fmaf(pq[(size_t)i * r + f], S[(size_t)f * (dv + 1) + dv], den);
        if (causal)
            for (int j = 0; j <= i; ++j) den += A[i][j];
        den_s[i] = den;
    }
    __syncthreads();
    // warp per row: lanes over value columns
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int i = warp; i < n; i += nw) {
        const float den = den_s[i];
        float gdo = 0.f;
        for (int c = lane; c < dv; c += 32) {
            float num = 0.f;
            for (int f = 0; f < r; ++f) num = fmaf(pq[(size_t)i * r + f], S[(size_t)f * (dv + 1) + c], num);
            if (causal)
                for (int j = 0; j <= i; ++j) num = fmaf(A[i][j], load_in(vb, (size_t)j * dv + c), num);
            const float gi = g[((size_t)bh * L + t0 + i) * dv + c];
            gdo = fmaf(gi, num / den, gdo);
            Y[((size_t)bh * L + t0 + i) * (dv + 1) + c] = gi / den;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) gdo += __shfl_xor_sync(0xffffffffu, gdo, o);
        if (lane == 0) Y[((size_t)bh * L + t0 + i) * (dv + 1) + dv] = -gdo / den;
    }
}

// per segment: R[f][c] = sum_{rows} phi_q[row][f] Y[row][c], c <= dv.
// grid (ceil(r/32), dv+1, BH*nseg), 32 threads.
__global__ void bwd_state(const float *__restrict__ phiq, const float *__restrict__ Y, float *__restrict__ R, int L,
                          int r, int dv, int seg, int nseg) {
    const int f = blockIdx.x * 32 + threadIdx.x, c = blockIdx.y;
    const int bh = blockIdx.z / nseg, s = blockIdx.z % nseg;
    if (f >= r) return;
    const int t0 = s * seg, t1 = min(L, t0 + seg);
    float acc = 0.f;
    for (int t = t0; t < t1; ++t)
        acc = fmaf(phiq[((size_t)bh * L + t) * r + f], Y[((size_t)bh * L + t) * (dv + 1) + c], acc);
    R[(((size_t)bh * nseg + s) * r + f) * (dv + 1) + c] = acc;
}

// exclusive suffix over segments, in place: R_s <- sum_{s' > s} R_s'
__global__ void bwd_state_suffix(float *__restrict__ R, int nseg, size_t per_seg, int BH) {
    const size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (e >= per_seg * BH) return;
    const int bh = (int)(e / per_seg);
    const size_t within = e % per_seg;
    float run = 0.f;
    for (int s = nseg - 1; s >= 0; --s) {
        float *p = R + ((size_t)bh * nseg + s) * per_seg + within;
        const float t = *p;
        *p = run;
        run += t;
    }
}

// dphi_q, dphi_k [rows][r] and dv [rows][dv] of a chunk from the entering
// state S, the leaving state R and (causal) the masked A, B inside it.
// block per (chunk, head), 256 threads.
template <typename T>
__global__ void bwd_chunk(const float *__restrict__ phiq, const float *__restrict__ phik, const T *__restrict__ v,
                          const float *__restrict__ Sin, const float *__restrict__ Rout, const float *__restrict__ Y,
                          float *__restrict__ dphiq, float *__restrict__ dphik, float *__restrict__ dV, int L, int r,
                          int dv, int nst, int causal) {
    __shared__ float A[kBwdRows][kBwdRows + 1];
    __shared__ float Bm[kBwdRows][kBwdRows + 1];
    const int ch = blockIdx.x, bh = blockIdx.y, t0 = ch * kBwdRows, n = min(kBwdRows, L - t0);
    const size_t row0 = (size_t)bh * L + t0;
    const float *pq = phiq + row0 * r, *pk = phik + row0 * r, *y = Y + row0 * (dv + 1);
    const T *vb = v + row0 * dv;
    const size_t st = ((size_t)bh * nst + (causal ? ch : 0)) * r * (dv + 1);
    const float *S = Sin + st, *R = Rout + st;
    if (causal) {
        for (int e = threadIdx.x; e < kBwdRows * kBwdRows; e += blockDim.x) {
            const int i = e / kBwdRows, j = e % kBwdRows;
            float a = 0.f, b = 0.f;
            if (i < n && j <= i) {
                for (int f = 0; f < r; ++f) a = fmaf(pq[(size_t)i * r + f], pk[(size_t)j * r + f], a);
                b = y[(size_t)i * (dv + 1) + dv];
                for (int c = 0; c < dv; ++c) b = fmaf(y[(size_t)i * (dv + 1) + c], load_in(vb, (size_t)j * dv + c), b);
            }
            A[i][j] = a;
            Bm[i][j] = b;
        }
        __syncthreads();
    }
    for (int e = threadIdx.x; e < n * r; e += blockDim.x) {
        const int i = e / r, f = e % r;
        // dphi_q[i][f] = S_f . dnum_i + z_f dden_i + sum_{j <= i} B_ij phi_k[j][f]
        float aq = S[(size_t)f * (dv + 1) + dv] * y[(size_t)i * (dv + 1) + dv];
        for (int c = 0; c < dv; ++c) aq = fmaf(S[(size_t)f * (dv + 1) + c], y[(size_t)i * (dv + 1) + c], aq);
        // dphi_k[i][f] = R_f . v_i + rho_f + sum_{i' >= i} B_i'i phi_q[i'][f]
        float ak = R[(size_t)f * (dv + 1) + dv];
        for (int c = 0; c < dv; ++c) ak = fmaf(R[(size_t)f * (dv + 1) + c], load_in(vb, (size_t)i * dv + c), ak);
        if (causal) {
            for (int j = 0; j <= i; ++j) aq = fmaf(Bm[i][j], pk[(size_t)j * r + f], aq);
            for (int j = i; j < n; ++j) ak = fmaf(Bm[j][i], pq[(size_t)j * r + f], ak);
        }
        dphiq[(row0 + i) * r + f] = aq;
        dphik[(row0 + i) * r + f] = ak;
    }
    for (int e = threadIdx.x; e < n * dv; e += blockDim.x) {
        const int j = e / dv, c = e % dv;
        // dv[j][c] = R[:, c] . phi_k[j] + sum_{i >= j} A_ij dnum_i[c]
        float acc = 0.f;
        for (int f = 0; f < r; ++f) acc = fmaf(R[(size_t)f * (dv + 1) + c], pk[(size_t)j * r + f], acc);
        if (causal)
            for (int i = j; i < n; ++i) acc = fmaf(A[i][j], y[(size_t)i * (dv + 1) + c], acc);
        dV[(row0 + j) * dv + c] = acc;
    }
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

// dx [rows][d] from the coefficients: warp per row, lanes over d
template <typename T>
__global__ void bwd_dx(const float *__restrict__ C, const float *__restrict__ dphi, const float *__restrict__ phi,
                       const T *__restrict__ x, const float *__restrict__ omega, float *__restrict__ dx, size_t rows,
                       int L, int H, int d, int nproj, int r, int map) {
    const size_t row = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float *c = C + row * nproj;
    if (map_is_elementwise(map)) {
        for (int j = lane; j < d; j += 32) dx[row * d + j] = c[j];
        return;
    }
    const int h = (int)((row / L) % H);
    const float *w = omega + (size_t)h * nproj * d;
    float tot = 0.f;
    if (map == FAVOR_MAP_POSITIVE) {
        for (int p = lane; p < nproj; p += 32) tot += c[p];
    } else if (map == FAVOR_MAP_TRIG_SOFTMAX) {
        for (int f = lane; f < r; f += 32) tot = fmaf(dphi[row * r + f], phi[row * r + f], tot);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    for (int j = lane; j < d; j += 32) {
        float acc = 0.f;
        for (int p = 0; p < nproj; ++p) acc = fmaf(c[p], w[(size_t)p * d + j], acc);
        const float xj = load_in(x, row * d + j);
        if (map == FAVOR_MAP_POSITIVE) acc = fmaf(-tot, xj, acc);
        else if (map == FAVOR_MAP_TRIG_SOFTMAX) acc = fmaf(tot, xj, acc);
        dx[row * d + j] = acc;
    }
}

// dw[h][p][j] += sum over a slice of the head's rows (all batches, queries
// and keys) of c[row][p] x[row][j]; grid (ceil(nproj d / 256), H, slices)
template <typename T>
__global__ void bwd_dw(const float *__restrict__ Cq, const float *__restrict__ Ck, const T *__restrict__ q,
                       const T *__restrict__ k, float *__restrict__ dw, int B, int H, int L, int d, int nproj,
                       int slice) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x, h = blockIdx.y;
    if (e >= nproj * d) return;
    const int p = e / d, j = e % d;
    const int r0 = blockIdx.z * slice, r1 = min(B * L, r0 + slice);
    float acc = 0.f;
    for (int t = r0; t < r1; ++t) {
        const int b = t / L, i = t % L;
        const size_t row = ((size_t)b * H + h) * L + i;
        acc = fmaf(Cq[row * nproj + p], load_in(q, row * d + j), acc);
        acc = fmaf(Ck[row * nproj + p], load_in(k, row * d + j), acc);
    }
    atomicAdd(&dw[((size_t)h * nproj + p) * d + j], acc);
}

template <typename T>
int backward_t(const T *q, const T *k, const T *v, const float *omega, const float *g, float *dq, float *dk,
               float *dv, float *dw, const Problem &p, cudaStream_t st) {
    const size_t rows = (size_t)p.BH * p.L;
    const int nch = p.causal ? (p.L + kBwdRows - 1) / kBwdRows : 1;
    const int seg = p.causal ? kBwdRows : p.L;
    const size_t per = (size_t)p.r * (p.dv + 1);
    size_t bytes = 2 * carve_bytes<float>(rows * p.nproj) + 4 * carve_bytes<float>(rows * p.r) +
                   2 * carve_bytes<float>(rows) + carve_bytes<float>(p.BH) +
                   2 * carve_bytes<float>((size_t)p.BH * nch * per) + carve_bytes<float>(rows * (p.dv + 1));
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
    float *Y = cv.take<float>(rows * (p.dv + 1));

    int rc;
    if ((rc = features_into<T>(q, omega, Pq, phiq, lsq, p, st)) || (rc = features_into<T>(k, omega, Pk, phik, lsk, p, st)))
        return rc;
    simt_head_max<<<p.BH, 256, 0, st>>>(lsk, hmax, p.L);
    FAVOR_LAUNCH_CHECK();
    const size_t total = rows * p.r;
    const unsigned sg = (unsigned)std::min<size_t>((total + 255) / 256, 152 * 64);
    simt_key_scale<<<sg, 256, 0, st>>>(phik, lsk, hmax, p.L, p.r, total);
    FAVOR_LAUNCH_CHECK();
    // the forward states entering each chunk (causal) or the total
    simt_state<T><<<dim3((p.r + 31) / 32, p.dv + 1, p.BH * nch), 32, 0, st>>>(phik, v, S, p.L, p.r, p.dv, seg, nch);
    FAVOR_LAUNCH_CHECK();
    if (p.causal) {
        simt_state_prefix<<<(unsigned)((per * p.BH + 255) / 256), 256, 0, st>>>(S, nch, per, p.BH);
        FAVOR_LAUNCH_CHECK();
    }
    const dim3 cg((p.L + kBwdRows - 1) / kBwdRows, p.BH);
    bwd_rows<T><<<cg, 256, 0, st>>>(phiq, phik, v, S, g, Y, p.L, p.r, p.dv, nch, p.causal);
    FAVOR_LAUNCH_CHECK();
    // the states leaving each chunk: exclusive suffix (causal) or the total
    bwd_state<<<dim3((p.r + 31) / 32, p.dv + 1, p.BH * nch), 32, 0, st>>>(phiq, Y, R, p.L, p.r, p.dv, seg, nch);
    FAVOR_LAUNCH_CHECK();
    if (p.causal) {
        bwd_state_suffix<<<(unsigned)((per * p.BH + 255) / 256), 256, 0, st>>>(R, nch, per, p.BH);
        FAVOR_LAUNCH_CHECK();
    }
    stats_begin(st, "bwd_chunk");
    bwd_chunk<T><<<cg, 256, 0, st>>>(phiq, phik, v, S, R, Y, dphiq, dphik, dv, p.L, p.r, p.dv, nch, p.causal);
    stats_end(st);
    FAVOR_LAUNCH_CHECK();
    const unsigned cgr = (unsigned)std::min<size_t>((rows * p.nproj + 255) / 256, 152 * 64);
    bwd_coeff<<<cgr, 256, 0, st>>>(Pq, dphiq, phiq, lsq, hmax, rows, p.L, p.nproj, p.r, p.map, 0);
    FAVOR_LAUNCH_CHECK();
    bwd_coeff<<<cgr, 256, 0, st>>>(Pk, dphik, phik, lsk, hmax, rows, p.L, p.nproj, p.r, p.map, 1);
    FAVOR_LAUNCH_CHECK();
    const unsigned xg = (unsigned)((rows * 32 + 255) / 256);
    bwd_dx<T><<<xg, 256, 0, st>>>(Pq, dphiq, phiq, q, omega, dq, rows, p.L, p.H, p.d, p.nproj, p.r, p.map);
    FAVOR_LAUNCH_CHECK();
    bwd_dx<T><<<xg, 256, 0, st>>>(Pk, dphik, phik, k, omega, dk, rows, p.L, p.H, p.d, p.nproj, p.r, p.map);
    FAVOR_LAUNCH_CHECK();
    if (dw && !map_is_elementwise(p.map)) {
        if (cudaMemsetAsync(dw, 0, (size_t)p.H * p.nproj * p.d * sizeof(float), st) != cudaSuccess) return FAVOR_ERR_CUDA;
        const int brows = p.B * p.L, slices = std::max(1, std::min(64, brows / 256));
        const int slice = (brows + slices - 1) / slices;
        bwd_dw<T><<<dim3((p.nproj * p.d + 255) / 256, p.H, slices), 256, 0, st>>>(Pq, Pk, q, k, dw, p.B, p.H, p.L,
                                                                                  p.d, p.nproj, slice);
        FAVOR_LAUNCH_CHECK();
    }
    return FAVOR_OK;
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

}  // namespace favor
