// favor_omega.cu -- the random projections w_i drawn on the device, for
// callers that redraw them (per step or per layer) without a host round trip.
//
// The pages draw w_i ~ N(0, I_d) ("Performer: Unbiased Softmax
// Approximation", the w ~ N(0, I) draw) and name orthogonal random features
// as the lower-variance variant (Performer study notes); they leave the
// generator open.  The draw here is fixed completely, so that any
// implementation reproduces it:
//   Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
//     Easy as 1, 2, 3", SC 2011) under key (seed, 0);
//   normal number e of stream s: the block at counter (e / 4, s, 0, 0), words
//     (x0, x1) -> normals 0, 1 and (x2, x3) -> normals 2, 3 by Box-Muller with
//     u = (x / 2^11 + 1/2) 2^-53, in fp64;
//   iid:        omega[h][i][j] = normal (h m + i) d + j of stream 0;
//   orthogonal: per head ceil(m / d) blocks; block b is the d x d matrix of
//     normals ((h nb + b) d + i) d + j of stream 0, its rows orthonormalised
//     by modified Gram-Schmidt in row order, row i scaled by the norm of
//     normals ((h nb + b) d + i) d + t (t < d) of stream 1; the last block
//     is truncated to the remaining rows.
// The kernels compute in fp64 and round the result to fp32 once.
#include <algorithm>

#include "favor_internal.h"

namespace favor {
namespace {

__device__ __forceinline__ void philox4x64_10(uint64_t (&c)[4], uint64_t k0, uint64_t k1) {
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += W0;
            k1 += W1;
        }
        const uint64_t hi0 = __umul64hi(M0, c[0]), lo0 = M0 * c[0];
        const uint64_t hi1 = __umul64hi(M1, c[2]), lo1 = M1 * c[2];
        const uint64_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
    }
}

// the four normals of block q of a stream
__device__ __forceinline__ void normals4(uint64_t seed, uint64_t stream, uint64_t q, double (&z)[4]) {
    uint64_t c[4] = {q, stream, 0, 0};
    philox4x64_10(c, seed, 0);
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const double u1 = ((double)(c[2 * p] >> 11) + 0.5) * 0x1p-53;
        const double u2 = ((double)(c[2 * p + 1] >> 11) + 0.5) * 0x1p-53;
        const double rad = sqrt(-2.0 * log(u1)), ang = 2.0 * 3.14159265358979323846 * u2;
        z[2 * p] = rad * cos(ang);
        z[2 * p + 1] = rad * sin(ang);
    }
}

__global__ void omega_iid(float *__restrict__ omega, uint64_t total, uint64_t seed) {
    for (uint64_t q = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; 4 * q < total;
         q += (uint64_t)gridDim.x * blockDim.x) {
        double z[4];
        normals4(seed, 0, q, z);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (4 * q + i < total) omega[4 * q + i] = __double2float_rn(z[i]);
    }
}

constexpr int kOrthThreads = 256;

// sum of a warp's values, the same on every lane
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// The normals of every block (stream 0, into Gall [H nb][d][d]) and the row
// norms' chi(d) factors (d normals of stream 1 per row, into chi [H nb][d]),
// over the whole GPU: fp64 transcendentals are the costly part of the draw.
__global__ void omega_orth_normals(double *__restrict__ Gall, double *__restrict__ chi, int H, int nb, int m,
                                   int d, uint64_t seed) {
    const uint64_t total4 = (uint64_t)H * nb * d * d / 4;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t q = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; q < total4; q += stride) {
        double z[4];
        normals4(seed, 0, q, z);
#pragma unroll
        for (int i = 0; i < 4; ++i) Gall[4 * q + i] = z[i];
    }
    const int lane = threadIdx.x & 31;
    const uint64_t nrows = (uint64_t)H * nb * d;
    for (uint64_t row = (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x) >> 5; row < nrows; row += stride >> 5) {
        if ((int)((row / d) % nb) * d + (int)(row % d) >= m) continue;   // past the truncation
        double ss = 0.0;
        for (int q = lane; q < d / 4; q += 32) {
            double z[4];
            normals4(seed, 1, row * d / 4 + q, z);
#pragma unroll
            for (int k = 0; k < 4; ++k) ss = fma(z[k], z[k], ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) chi[row] = sqrt(ss);
    }
}

// grid (blocks per head, H): one d x d block of one head
__global__ void __launch_bounds__(kOrthThreads) omega_orth(float *__restrict__ omega, const double *__restrict__ Gall,
                                                            const double *__restrict__ chi_all, int m, int d) {
    extern __shared__ double G[];           // [d][d]
    const int b = blockIdx.x, h = blockIdx.y, nb = gridDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarp = kOrthThreads / 32;
    const size_t blk = (size_t)h * nb + b;
    const int rows = min(d, m - b * d);
    const double *chi = chi_all + blk * d;
    for (int e = tid; e < rows * d; e += kOrthThreads) G[e] = Gall[blk * d * d + e];
    __syncthreads();
    // modified Gram-Schmidt, right-looking: once row j is normalised, every
    // later row loses its component along it (row i sees q_0, q_1, ... in the
    // order the row-by-row form applies them)
    // (rows past the truncation are never needed: a row depends only on the
    // rows before it)
    for (int j = 0; j < rows; ++j) {
        double *qj = G + (size_t)j * d;
        if (warp == 0) {
            double ss = 0.0;
            for (int t = lane; t < d; t += 32) ss = fma(qj[t], qj[t], ss);
            const double nrm = sqrt(warp_sum(ss));
            for (int t = lane; t < d; t += 32) qj[t] /= nrm;
        }
        __syncthreads();
        for (int i = j + 1 + warp; i < rows; i += nwarp) {
            double *v = G + (size_t)i * d;
            double dot = 0.0;
            for (int t = lane; t < d; t += 32) dot = fma(v[t], qj[t], dot);
            dot = warp_sum(dot);
            for (int t = lane; t < d; t += 32) v[t] -= dot * qj[t];
        }
        __syncthreads();
    }
    float *dst = omega + ((size_t)h * m + (size_t)b * d) * d;
    for (int e = tid; e < rows * d; e += kOrthThreads) dst[e] = __double2float_rn(G[e] * chi[e / d]);
}

}  // namespace
}  // namespace favor

using namespace favor;

extern "C" int favor_draw_omega(float *omega, int H, int m, int d, int kind, unsigned long long seed,
                                cudaStream_t stream) {
    if (H < 1 || m < 1 || (kind != 0 && kind != 1)) return FAVOR_ERR_INVALID_ARG;
    if (d != 32 && d != 64 && d != 128) return FAVOR_ERR_UNSUPPORTED;
    if ((long long)H * m * d > (1ll << 40)) return FAVOR_ERR_UNSUPPORTED;
    int rc;
    if ((rc = check_ptr(omega, false))) return rc;
    const uint64_t total = (uint64_t)H * m * d;
    if (kind == 0) {
        const uint64_t blocks = (total / 4 + 255) / 256;
        omega_iid<<<(unsigned)std::min<uint64_t>(blocks, 152 * 16), 256, 0, stream>>>(omega, total, seed);
        FAVOR_LAUNCH_CHECK();
        return FAVOR_OK;
    }
    const int nb = (m + d - 1) / d;
    const size_t nG = (size_t)H * nb * d * d, nchi = (size_t)H * nb * d;
    int status = FAVOR_OK;
    void *ws = workspace(carve_bytes<double>(nG) + carve_bytes<double>(nchi), &status);
    if (!ws) return status;
    Carve cv{static_cast<char *>(ws), 0};
    double *Gall = cv.take<double>(nG), *chi = cv.take<double>(nchi);
    omega_orth_normals<<<152 * 8, 256, 0, stream>>>(Gall, chi, H, nb, m, d, seed);
    FAVOR_LAUNCH_CHECK();
    const size_t smem = (size_t)d * d * sizeof(double);
    if (cudaFuncSetAttribute(omega_orth, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return FAVOR_ERR_CUDA;
    }
    omega_orth<<<dim3(nb, H), kOrthThreads, smem, stream>>>(omega, Gall, chi, m, d);
    FAVOR_LAUNCH_CHECK();
    return FAVOR_OK;
}
