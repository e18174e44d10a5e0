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

}  // namespace favor
