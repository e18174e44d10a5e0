// favor_decode.cu -- the carried state of a key sequence and the one-token
// decode step.
//
// The causal form keeps running sums (Performer study notes, "Case 2"):
//   S_i = S_{i-1} + phi(k_i) v_i^T,  z_i = z_{i-1} + phi(k_i),
//   out_i = phi(q_i)^T S_i / phi(q_i)^T z_i        (diagonal j = i included)
// so a new token costs O(r d) against the stored (S, z) instead of a pass
// over the whole prefix.  phi is the feature map of the pages: positive
// exp(w.x - |x|^2/2)/sqrt(m) ("Kernel Feature Maps" section 4), trig
// (sin, cos)(w.x)/sqrt(m) interleaved per projection (section 3), elu1
// (section 1).
//
// Decode state of one head (b, h): r (dv + 2) fp32 values
//   S^ [r][dv] | z^ [r] | rho [r]
// with S_f = S^_f 2^rho_f and z_f = z^_f 2^rho_f.  rho_f is a per-feature
// log2 reference: a step raises it to the new key's log2 feature when that is
// larger and rescales the row, so every stored value stays within fp32 range
// whatever the size of the exponents.  An empty state has S^ = z^ = 0 and
// rho = -inf.
//
// Kernels:
//   decode_export  piece states of the state pass -> decode state
//   decode_empty   the empty state
//   decode_step    one token per head: persistent CTAs stream the state
//                  through a ring of shared-memory stages filled by bulk
//                  copies.  The step reads and writes the state once: it is
//                  bound by HBM (or by launch latency for small batches), so
//                  it is plain SIMT arithmetic in fp32.
#include <cmath>

#include <algorithm>

#include "favor_internal.h"
#include "tc_ptx.cuh"

namespace favor {
namespace {

using namespace tc;

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float load_in(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_in(const uint16_t *p, size_t i) {
    return __uint_as_float(static_cast<uint32_t>(p[i]) << 16);
}

// ---------------------------------------------------------------------------
// decode_export: per head, the pieces' rows summed in piece order at the
// largest of their references; block = 8 features x 32 column threads.
// ---------------------------------------------------------------------------
struct ExportArgs {
    const float *src;   // [BH][np][r][dv + 1]
    const float *ref;   // reference of (piece g, tile t): ref[((bh np + g) nrt + t) rstride]
    int np, nrt, rstride, r, dv;
    float ref_scale;    // rho = ref_scale R* + rho_add (log2 units)
    float rho_add;
    int trig_tiles;     // source trig features in 128-column tiles [sin 64 | cos 64]
    float *state;       // [BH][r (dv + 2)]
};

constexpr int kMaxPieces = 64;

__global__ void decode_export(const ExportArgs a) {
    __shared__ float sc[8][kMaxPieces];
    __shared__ float rstar[8];
    const int bh = blockIdx.y, fl = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int fs = blockIdx.x * 8 + fl;
    const bool valid = fs < a.r;
    const int t = a.nrt > 1 ? fs / 128 : 0;
    auto ref_of = [&](int g) { return a.ref[(((size_t)bh * a.np + g) * a.nrt + t) * a.rstride]; };
    if (valid) {
        float R = -INFINITY;
        for (int g = lane; g < a.np; g += 32) R = fmaxf(R, ref_of(g));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) R = fmaxf(R, __shfl_xor_sync(0xffffffffu, R, o));
        for (int g = lane; g < a.np; g += 32) {
            const float Rg = ref_of(g);
            sc[fl][g] = (Rg == -INFINITY || R == -INFINITY) ? 0.f : exp2f(Rg - R);
        }
        if (lane == 0) rstar[fl] = R;
    }
    __syncthreads();
    if (!valid) return;
    int fd = fs;
    if (a.trig_tiles) {
        const int c = fs % 128, proj = (fs / 128) * 64 + (c & 63);
        fd = 2 * proj + (c >= 64 ? 1 : 0);
    }
    const size_t W = (size_t)a.dv + 1;
    float *dst = a.state + (size_t)bh * a.r * (a.dv + 2);
    for (int c = lane; c <= a.dv; c += 32) {
        float sum = 0.f;
        for (int g = 0; g < a.np; ++g)
            sum = fmaf(a.src[(((size_t)bh * a.np + g) * a.r + fs) * W + c], sc[fl][g], sum);
        if (c < a.dv) dst[(size_t)fd * a.dv + c] = sum;
        else dst[(size_t)a.r * a.dv + fd] = sum;
    }
    if (lane == 0) dst[(size_t)a.r * (a.dv + 1) + fd] = a.ref_scale * rstar[fl] + a.rho_add;
}

__global__ void decode_empty(float *state, int r, int dv, size_t total) {
    const size_t per = (size_t)r * (dv + 2);
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
         e += (size_t)gridDim.x * blockDim.x)
        state[e] = (e % per) >= (size_t)r * (dv + 1) ? -INFINITY : 0.f;
}

// ---------------------------------------------------------------------------
// decode_step: persistent CTAs (256 threads), each on the heads b, b + grid,
// ... of the batch, a head as ceil(r / 64) tiles of 64 features.  Thread 0
// streams tiles into a ring of shared-memory stages with bulk copies (the
// tile's rows of S^, its z^ and rho, and the head's q, k, v), running up to
// a ring's length ahead across heads; every thread then
//   A  as (f, s) = (tid / 4, tid % 4): the projections of feature f from a
//      quarter of d each, then the feature's raised reference, rescale alpha,
//      key weight p, query weight and new z^ (s = 0 stores z^ and rho);
//   B  as (g, c) = (tid / dv, tid % dv): value column c of the rows of
//      feature group g (dv / 4 features): the updated S^ (stored) and its
//      query-weighted sum.
// The numerator and denominator of a head are summed over its tiles at a
// running maximum of the query's log2 weights.  The step streams the state
// once each way: an HBM-bound kernel in fp32 SIMT arithmetic.
// ---------------------------------------------------------------------------
struct DecodeArgs {
    const void *q, *k, *v;   // [BH][d], [BH][d], [BH][dv]
    const float *omega;      // [H][m][d] (unused for elu1)
    float *state;            // [BH][r (dv + 2)]
    float *out;              // [BH][dv]
    int *status;
    int BH, H, d, dv, m, r, map, esize;
    int cph;                 // CTAs per head (a cluster), or 1: persistent CTAs over heads
};

constexpr int kDecFt = 64;                  // features per tile
constexpr int kDecThreads = 4 * kDecFt;
constexpr int kDecStages = 4;
constexpr int kDecWarps = kDecThreads / 32;
constexpr long long kDecWaitLimit = 1ll << 32;

// stage layout (bytes): S^ rows [64][dv] fp32 | z^ [64] | rho [64] | q | k | v
// (q, k, v in the input type, 512 bytes each at most)
__host__ __device__ constexpr uint32_t dec_stage_bytes(int dv) { return (uint32_t)kDecFt * dv * 4 + 2048; }

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// generic address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ const float *cluster_map(const float *p, uint32_t rank) {
    uint64_t out;
    asm volatile("mapa.u64 %0, %1, %2;" : "=l"(out) : "l"(p), "r"(rank));
    return reinterpret_cast<const float *>(out);
}

template <typename T, int D, int DV>
__global__ void __launch_bounds__(kDecThreads) decode_step(const DecodeArgs a) {
    constexpr int FPG = DV / 4;             // features per phase-B group
    constexpr int DD = D / 4, NW4 = DD / 4;  // d per phase-A thread, its float4s of w
    constexpr uint32_t SB = dec_stage_bytes(DV);
    constexpr uint32_t OZ = kDecFt * DV * 4, ORHO = OZ + 256, OQ = OZ + 512, OK = OZ + 1024, OV = OZ + 1536;
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ uint64_t full[kDecStages];
    __shared__ float s_alpha[kDecFt], s_p[kDecFt], s_w[kDecFt];
    __shared__ float wmax[kDecWarps], wden[kDecWarps];
    __shared__ float red[kDecThreads];
    __shared__ float part[2 + DV];          // (max, den, num[DV]) of a head's tiles in this CTA
    __shared__ int abort_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = a.r;
    const int nt = (r + kDecFt - 1) / kDecFt;
    // the CTA's heads and tiles: with cph > 1 the CTAs of a cluster share one
    // head, CTA j taking tiles j, j + cph, ...; else heads b, b + grid, ...
    const int cph = a.cph, rank = cph > 1 ? (int)(blockIdx.x % cph) : 0;
    const int hb = cph > 1 ? (int)(blockIdx.x / cph) : (int)blockIdx.x;
    const int hstride = cph > 1 ? a.BH : (int)gridDim.x;
    const int ntc = (nt - rank + cph - 1) / cph;    // tiles per head here
    const int nheads = a.BH > hb ? (a.BH - 1 - hb) / hstride + 1 : 0;
    const int total = nheads * ntc;
    const size_t per_head = (size_t)r * (DV + 2);

    auto head_of = [&](int n) { return hb + (n / ntc) * hstride; };
    auto tile_of = [&](int n) { return rank + (n % ntc) * cph; };
    // thread 0: bulk copies of tile n into stage n % stages
    auto issue = [&](int n) {
        const int bh = head_of(n), t = tile_of(n), f0 = t * kDecFt, nf = min(kDecFt, r - f0);
        uint8_t *sg = dsm + (size_t)(n % kDecStages) * SB;
        const float *src = a.state + (size_t)bh * per_head;
        const uint32_t sbytes = (uint32_t)nf * DV * 4, vbytes = (uint32_t)nf * 4;
        const uint32_t xb = (uint32_t)D * a.esize, vb = (uint32_t)DV * a.esize;
        uint64_t *bar = &full[n % kDecStages];
        mbar_arrive_expect_tx(bar, sbytes + 2 * vbytes + 2 * xb + vb);
        bulk_load(sg, src + (size_t)f0 * DV, sbytes, bar);
        bulk_load(sg + OZ, src + (size_t)r * DV + f0, vbytes, bar);
        bulk_load(sg + ORHO, src + (size_t)r * (DV + 1) + f0, vbytes, bar);
        bulk_load(sg + OQ, static_cast<const uint8_t *>(a.q) + (size_t)bh * xb, xb, bar);
        bulk_load(sg + OK, static_cast<const uint8_t *>(a.k) + (size_t)bh * xb, xb, bar);
        bulk_load(sg + OV, static_cast<const uint8_t *>(a.v) + (size_t)bh * vb, vb, bar);
    };

    if (tid == 0) {
        for (int i = 0; i < kDecStages; ++i) mbar_init(&full[i], 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();
    if (tid == 0)
        for (int n = 0; n < min(kDecStages, total); ++n) issue(n);

    const int fl = tid >> 2, s = tid & 3;           // phase A
    const int g = tid / DV, c = tid % DV;           // phase B
    const float half_log2m = 0.5f * log2f((float)a.m);
    // this thread's quarter of the projection row of tile n's feature
    auto load_w = [&](int n, float4 (&w)[NW4]) {
        const int f = tile_of(n) * kDecFt + fl;
        if (map_is_elementwise(a.map) || f >= r) return;
        const int p = map_is_trig(a.map) ? f >> 1 : f;
        const float4 *w4 =
            reinterpret_cast<const float4 *>(a.omega + ((size_t)(head_of(n) % a.H) * a.m + p) * D + s * DD);
#pragma unroll
        for (int i = 0; i < NW4; ++i) w[i] = w4[i];
    };
    float4 wv[NW4], wn[NW4];
#pragma unroll
    for (int i = 0; i < NW4; ++i) wn[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (total > 0) load_w(0, wn);
    float M = -INFINITY, den_acc = 0.f, num_acc = 0.f;
    int n = 0;
    for (; n < total; ++n) {
        const int bh = head_of(n), t = tile_of(n), f0 = t * kDecFt;
#pragma unroll
        for (int i = 0; i < NW4; ++i) wv[i] = wn[i];
        const uint8_t *sg = dsm + (size_t)(n % kDecStages) * SB;
        const float *S_t = reinterpret_cast<const float *>(sg);
        const float *z_t = reinterpret_cast<const float *>(sg + OZ);
        const float *rho_t = reinterpret_cast<const float *>(sg + ORHO);
        const T *xq = reinterpret_cast<const T *>(sg + OQ);
        const T *xk = reinterpret_cast<const T *>(sg + OK);
        const T *xv = reinterpret_cast<const T *>(sg + OV);
        float *st = a.state + (size_t)bh * per_head;
        // bounded wait for the stage (another thread's timeout ends it too)
        bool ok = mbar_try_wait(&full[n % kDecStages], (n / kDecStages) & 1);
        if (!ok) {
            const long long t0 = clock64();
            while (!(ok = mbar_try_wait(&full[n % kDecStages], (n / kDecStages) & 1))) {
                if (*static_cast<volatile int *>(&abort_flag)) break;
                if (clock64() - t0 > kDecWaitLimit) {
                    abort_flag = 1;
                    break;
                }
            }
        }
        // ---- phase A: feature f0 + fl
        const int f = f0 + fl;
        const bool valid = ok && f < r;
        float dq = 0.f, dk = 0.f, ss = 0.f;
        if (ok) {
            if (a.map == FAVOR_MAP_POSITIVE || a.map == FAVOR_MAP_TRIG_SOFTMAX) {
#pragma unroll
                for (int i = 0; i < DD; ++i) {
                    const float x = load_in(xk, s * DD + i);
                    ss = fmaf(x, x, ss);
                }
            }
            if (!map_is_elementwise(a.map) && valid) {
#pragma unroll
                for (int i = 0; i < NW4; ++i) {
                    const float4 w = wv[i];
                    const int j = s * DD + 4 * i;
                    dq = fmaf(w.x, load_in(xq, j), fmaf(w.y, load_in(xq, j + 1),
                         fmaf(w.z, load_in(xq, j + 2), fmaf(w.w, load_in(xq, j + 3), dq))));
                    dk = fmaf(w.x, load_in(xk, j), fmaf(w.y, load_in(xk, j + 1),
                         fmaf(w.z, load_in(xk, j + 2), fmaf(w.w, load_in(xk, j + 3), dk))));
                }
            }
        }
        dq += __shfl_xor_sync(0xffffffffu, dq, 1);
        dq += __shfl_xor_sync(0xffffffffu, dq, 2);
        dk += __shfl_xor_sync(0xffffffffu, dk, 1);
        dk += __shfl_xor_sync(0xffffffffu, dk, 2);
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);   // |k|^2: the quarters of a quad cover k
        // feature = raw value x 2^(log2 scale); the 1/sqrt(m) factor sits in
        // the key's scale (the query's per-row factors cancel in num / den)
        float ek = 0.f, pk = 1.f, eq = 0.f, pq = 1.f;
        if (a.map == FAVOR_MAP_POSITIVE) {
            ek = kLog2e * (dk - 0.5f * ss) - half_log2m;
            eq = kLog2e * dq;
        } else if (map_is_trig(a.map)) {
            float sn, cs;
            sincosf(dk, &sn, &cs);
            pk = (f & 1) ? cs : sn;
            sincosf(dq, &sn, &cs);
            pq = (f & 1) ? cs : sn;
            // the softmax-scaled map carries exp(|k|^2/2) in the key's scale
            ek = (a.map == FAVOR_MAP_TRIG_SOFTMAX ? 0.5f * kLog2e * ss : 0.f) - half_log2m;
        } else if (valid) {
            const float x = load_in(xk, f), y = load_in(xq, f);
            if (a.map == FAVOR_MAP_RELU) {
                pk = fmaxf(x, 0.f);
                pq = fmaxf(y, 0.f);
            } else {
                pk = x > 0.f ? x + 1.f : expf(x);
                pq = y > 0.f ? y + 1.f : expf(y);
            }
        }
        float sq = -INFINITY, zn = 0.f;
        if (valid) {
            const float rho = rho_t[fl];
            const float Rn = fmaxf(rho, ek);
            const float alpha = exp2f(rho - Rn), pw = pk * exp2f(ek - Rn);
            zn = fmaf(alpha, z_t[fl], pw);
            sq = eq + Rn;
            if (s == 0) {
                s_alpha[fl] = alpha;
                s_p[fl] = pw;
                st[(size_t)r * DV + f] = zn;
                st[(size_t)r * (DV + 1) + f] = Rn;
            }
        }
        // query weights relative to the warp's largest (8 features a warp)
        float mw = sq;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
        const float wq = valid ? pq * exp2f(sq - mw) : 0.f;
        float dsum = (s == 0) ? wq * zn : 0.f;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
        if (s == 0) s_w[fl] = wq;
        if (lane == 0) {
            wmax[warp] = mw;
            wden[warp] = dsum;
        }
        if (__syncthreads_or(!ok)) break;
        // the next tile's projection rows load while this one finishes
        if (n + 1 < total) load_w(n + 1, wn);
        // the tile's largest query weight; the running maximum of the head
        float mt = wmax[0];
#pragma unroll
        for (int i = 1; i < kDecWarps; ++i) mt = fmaxf(mt, wmax[i]);
        float den_t = 0.f;
#pragma unroll
        for (int i = 0; i < kDecWarps; ++i)
            if (wmax[i] != -INFINITY) den_t = fmaf(wden[i], exp2f(wmax[i] - mt), den_t);
        const float Mn = fmaxf(M, mt);
        const float sc_old = M == -INFINITY ? 0.f : exp2f(M - Mn), sc_new = exp2f(mt - Mn);
        M = Mn;
        den_acc = fmaf(den_acc, sc_old, den_t * sc_new);
        // ---- phase B: S^_f[c] <- alpha_f S^_f[c] + p_f v[c]; num[c] += w_f S^_f[c]
        {
            const float vc = load_in(xv, c);
            float num = 0.f;
#pragma unroll
            for (int j = 0; j < FPG; ++j) {
                const int flj = g * FPG + j, fj = f0 + flj;
                if (fj < r) {
                    const float x = fmaf(s_alpha[flj], S_t[flj * DV + c], s_p[flj] * vc);
                    st[(size_t)fj * DV + c] = x;
                    num = fmaf(s_w[flj] * exp2f(wmax[flj >> 3] - mt), x, num);
                }
            }
            num_acc = fmaf(num_acc, sc_old, num * sc_new);
        }
        const bool last = n % ntc == ntc - 1;
        if (last) red[tid] = num_acc;
        __syncthreads();
        if (last) {
            if (cph == 1) {
                if (tid < DV) {
                    float sum = 0.f;
                    for (int i = 0; i < kDecThreads / DV; ++i) sum += red[i * DV + tid];
                    a.out[(size_t)bh * DV + tid] = sum / den_acc;
                }
            } else {
                // the head's tiles are spread over the cluster: CTA 0 of the
                // cluster combines every CTA's (max, den, num)
                if (tid < DV) {
                    float sum = 0.f;
                    for (int i = 0; i < kDecThreads / DV; ++i) sum += red[i * DV + tid];
                    part[2 + tid] = sum;
                }
                if (tid == 0) {
                    part[0] = M;
                    part[1] = den_acc;
                }
                cluster_sync_all();
                if (rank == 0 && tid < DV) {
                    float Mt[4], dn[4], nm[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (j < cph) {
                            const float *pr = cluster_map(part, (uint32_t)j);
                            Mt[j] = pr[0];
                            dn[j] = pr[1];
                            nm[j] = pr[2 + tid];
                        }
                    float Mx = Mt[0];
#pragma unroll
                    for (int j = 1; j < 4; ++j)
                        if (j < cph) Mx = fmaxf(Mx, Mt[j]);
                    float num = 0.f, den = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (j < cph) {
                            const float sc = exp2f(Mt[j] - Mx);
                            num = fmaf(sc, nm[j], num);
                            den = fmaf(sc, dn[j], den);
                        }
                    a.out[(size_t)bh * DV + tid] = num / den;
                }
                // every CTA's part stays until CTA 0 has read it
                cluster_sync_all();
            }
            M = -INFINITY;
            den_acc = num_acc = 0.f;
        }
        // stage n % stages is free: refill it with the tile a ring further on
        if (tid == 0 && n + kDecStages < total) issue(n + kDecStages);
    }
    if (n < total) {
        // a wait ran out: record it, then let the copies in flight land
        // (bounded) before the CTA's shared memory goes away
        if (tid == 0) {
            atomicExch(a.status, FAVOR_ERR_TIMEOUT);
            for (int i = n; i < min(total, n + kDecStages); ++i) {
                const long long t0 = clock64();
                while (!mbar_try_wait(&full[i % kDecStages], (i / kDecStages) & 1) &&
                       clock64() - t0 < kDecWaitLimit) {
                }
            }
        }
        // a cluster's CTAs each pass its two barriers exactly once (the last
        // tile was not reached here), so that none of them waits forever
        if (cph > 1) {
            __syncthreads();
            cluster_sync_all();
            cluster_sync_all();
        }
    }
}

template <typename T, int D, int DV>
int decode_launch_t(const DecodeArgs &a0, cudaStream_t st) {
    const uint32_t smem = kDecStages * dec_stage_bytes(DV);
    auto kern = decode_step<T, D, DV>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return FAVOR_ERR_CUDA;
    }
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        return FAVOR_ERR_CUDA;
    }
    DecodeArgs a = a0;
    const int nt = (a.r + kDecFt - 1) / kDecFt;
    const int slots = std::max(1, sms) * std::max(1, per_sm);
    // fewer heads than CTA slots: a head's tiles over a cluster of up to 4 CTAs
    a.cph = 1;
    while (a.cph < 4 && 2 * a.cph <= nt && (long long)a.BH * 2 * a.cph <= slots) a.cph *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.cph > 1 ? a.BH * a.cph : std::min(a.BH, slots));
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = a.cph;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    stats_begin(st, "decode_step");
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
    stats_end(st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return FAVOR_ERR_CUDA;
    }
    stats_count_launch();
    return FAVOR_OK;
}

template <typename T, int D>
int decode_launch_d(const DecodeArgs &a, cudaStream_t st) {
    switch (a.dv) {
        case 32: return decode_launch_t<T, D, 32>(a, st);
        case 64: return decode_launch_t<T, D, 64>(a, st);
        default: return decode_launch_t<T, D, 128>(a, st);
    }
}

template <typename T>
int decode_launch(const DecodeArgs &a, cudaStream_t st) {
    switch (a.d) {
        case 32: return decode_launch_d<T, 32>(a, st);
        case 64: return decode_launch_d<T, 64>(a, st);
        default: return decode_launch_d<T, 128>(a, st);
    }
}

bool overlaps(const void *a, size_t an, const void *b, size_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a && b && a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace

int decode_state(const void *k, const void *v, bool bf16_in, const float *omega, float *state, int B,
                 int H, int L, int d, int dv, int m, int map, cudaStream_t st) {
    if (L < 0) return FAVOR_ERR_INVALID_ARG;
    Problem p;
    int rc = make_problem(B, H, L > 0 ? L : 1, d, dv, m, 1, map, &p);
    if (rc) return rc;
    if ((rc = check_ptr(state, false))) return rc;
    const size_t state_bytes = (size_t)p.BH * p.r * (p.dv + 2) * sizeof(float);
    if (L == 0) {
        const size_t total = state_bytes / sizeof(float);
        decode_empty<<<(unsigned)std::min<size_t>((total + 255) / 256, 4096), 256, 0, st>>>(state, p.r, p.dv,
                                                                                          total);
        FAVOR_LAUNCH_CHECK();
        return FAVOR_OK;
    }
    const size_t esize = bf16_in ? 2 : 4;
    if ((rc = check_ptr(k, false)) || (rc = check_ptr(v, false)) ||
        (rc = check_ptr(omega, map_is_elementwise(map))))
        return rc;
    const size_t rows = (size_t)p.BH * p.L;
    if (overlaps(state, state_bytes, k, rows * p.d * esize) || overlaps(state, state_bytes, v, rows * p.dv * esize) ||
        overlaps(state, state_bytes, omega, (size_t)p.H * p.nproj * p.d * sizeof(float)))
        return FAVOR_ERR_INVALID_ARG;
    ExportArgs ea{};
    ea.r = p.r;
    ea.dv = p.dv;
    ea.state = state;
    Problem pn = p;
    pn.causal = 0;
    if (bf16_in && tc_supported(pn)) {
        const float *src, *meta;
        int np;
        if ((rc = tc_key_state(k, v, omega, pn, st, &src, &meta, &np))) return rc;
        if (np > kMaxPieces) return FAVOR_ERR_UNSUPPORTED;
        ea.src = src;
        ea.ref = meta;
        ea.np = np;
        ea.nrt = (p.r + 127) / 128;
        ea.rstride = 4;
        ea.ref_scale = 1.f;
        ea.rho_add = map_is_elementwise(map) ? 0.f : -0.5f * log2f((float)p.m);
        ea.trig_tiles = map == FAVOR_MAP_TRIG;
    } else {
        const float *S, *hmax;
        if ((rc = simt_key_state(k, v, bf16_in, omega, pn, st, &S, &hmax))) return rc;
        ea.src = S;
        ea.ref = hmax;
        ea.np = 1;
        ea.nrt = 1;
        ea.rstride = 1;
        ea.ref_scale = kLog2e;
        ea.rho_add = 0.f;
        ea.trig_tiles = 0;
    }
    decode_export<<<dim3((p.r + 7) / 8, p.BH), 256, 0, st>>>(ea);
    FAVOR_LAUNCH_CHECK();
    return FAVOR_OK;
}

int decode_step_run(const void *q, const void *k, const void *v, bool bf16_in, const float *omega, float *state,
                    float *out, int B, int H, int d, int dv, int m, int map, cudaStream_t st) {
    Problem p;
    int rc = make_problem(B, H, 1, d, dv, m, 1, map, &p);
    if (rc) return rc;
    if (p.r > 1024) return FAVOR_ERR_UNSUPPORTED;
    if ((rc = check_ptr(q, false)) || (rc = check_ptr(k, false)) || (rc = check_ptr(v, false)) ||
        (rc = check_ptr(state, false)) || (rc = check_ptr(out, false)) ||
        (rc = check_ptr(omega, map_is_elementwise(map))))
        return rc;
    const size_t esize = bf16_in ? 2 : 4;
    const size_t sb = (size_t)p.BH * p.r * (p.dv + 2) * sizeof(float), ob = (size_t)p.BH * p.dv * sizeof(float);
    const size_t xb = (size_t)p.BH * p.d * esize, vb = (size_t)p.BH * p.dv * esize;
    const size_t wb = map_is_elementwise(map) ? 0 : (size_t)p.H * p.m * p.d * sizeof(float);
    const void *ins[4] = {q, k, v, omega};
    const size_t inb[4] = {xb, xb, vb, wb};
    for (int i = 0; i < 4; ++i)
        if (overlaps(state, sb, ins[i], inb[i]) || overlaps(out, ob, ins[i], inb[i])) return FAVOR_ERR_INVALID_ARG;
    if (overlaps(out, ob, state, sb)) return FAVOR_ERR_INVALID_ARG;
    DecodeArgs a;
    a.q = q; a.k = k; a.v = v; a.omega = omega; a.state = state; a.out = out;
    a.status = device_status_ptr();
    if (!a.status) return FAVOR_ERR_CUDA;
    a.BH = p.BH; a.H = p.H; a.d = p.d; a.dv = p.dv; a.m = p.m; a.r = p.r; a.map = map;
    a.esize = (int)esize;
    return bf16_in ? decode_launch<uint16_t>(a, st) : decode_launch<float>(a, st);
}

}  // namespace favor

using namespace favor;

extern "C" int favor_state_floats(int d, int dv, int m, int feature_map) {
    Problem p;
    if (make_problem(1, 1, 1, d, dv, m, 1, feature_map, &p)) return -1;
    return p.r * (p.dv + 2);
}

extern "C" int favor_attn_state(const void *k, const void *v, const float *omega, float *state, int B, int H,
                                int L, int d, int dv, int m, int feature_map, cudaStream_t stream) {
    return decode_state(k, v, true, omega, state, B, H, L, d, dv, m, feature_map, stream);
}

extern "C" int favor_attn_state_f32(const float *k, const float *v, const float *omega, float *state, int B,
                                    int H, int L, int d, int dv, int m, int feature_map, cudaStream_t stream) {
    return decode_state(k, v, false, omega, state, B, H, L, d, dv, m, feature_map, stream);
}

extern "C" int favor_attn_decode(const void *q, const void *k, const void *v, const float *omega, float *state,
                                 float *out, int B, int H, int d, int dv, int m, int feature_map,
                                 cudaStream_t stream) {
    return decode_step_run(q, k, v, true, omega, state, out, B, H, d, dv, m, feature_map, stream);
}

extern "C" int favor_attn_decode_f32(const float *q, const float *k, const float *v, const float *omega,
                                     float *state, float *out, int B, int H, int d, int dv, int m, int feature_map,
                                     cudaStream_t stream) {
    return decode_step_run(q, k, v, false, omega, state, out, B, H, d, dv, m, feature_map, stream);
}
