// favor_tc.cu -- the tensor-core path of the FAVOR+ forward pass on sm_103a.
//
// Per head (b, h) the path computes, in 128-token chunks:
//   features     phi(X) from the projection P = X W^T (tcgen05 MMA, TMA-fed,
//                fp32 accumulator in TMEM) and an exp / sin,cos / elu+1
//                epilogue that writes fp16 features to shared memory
//                ("Kernel Feature Maps" sections 1, 3, 4; Performer page phi(x))
//   state        S = phi(K)^T V and z = phi(K)^T 1 (tcgen05, fp32 in TMEM)
//   non-causal   out = phi(Q) S / phi(Q) z                (Performer page In[25])
//   causal       per chunk: A = phi(Q_c) phi(K_c)^T masked to j <= i,
//                num = A V_c + phi(Q_c) S, den = A 1 + phi(Q_c) z, then
//                S += phi(K_c)^T V_c                      (study notes, "Case 2")
//
// Stabilisers (they cancel exactly in num / den):
//   queries: each row is divided by exp(max_f w_f.q) and multiplied by e^8;
//   keys:    every key of a head shares one reference R (a running maximum of
//            w_f.k - |k|^2/2, raised only when a chunk exceeds it by more than
//            e^2; the state is rescaled when it moves), plus the same e^8.
// Those offsets keep every fp16 feature in [e^-20, e^10].  The intra-chunk
// matrix is normalised per row by a power of two before it is rounded to
// fp16, and the state operand by a power of two bounded from the running key
// mass; both factors are divided out in fp32.
//
// Kernels: tc_prep_omega (fp16 image of W), tc_state (segment states),
// tc_combine (fixed-order sums / exclusive prefixes of the segment states),
// tc_output (non-causal rows), tc_causal (the chunked causal scan).
#include <cmath>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "favor_internal.h"
#include "tc_ptx.cuh"

namespace favor {
namespace {

using namespace tc;

constexpr int kC = 128;                 // tokens per chunk (= MMA M)
constexpr int kThreads = 256;           // 8 warps: two per TMEM lane quarter
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kShift = 8.0f * 1.4426950408889634f;   // e^8 headroom (log2 units)
constexpr float kSlack = 2.0f * 1.4426950408889634f;   // tolerated excess before re-referencing
constexpr float kSigmaTarget = 16384.f;  // bound for |sigma * S| in the fp16 state operand
constexpr long long kWaitLimit = 1ll << 32;             // ~2 s of clock cycles
constexpr uint32_t kBlk = 16384;        // one [128][64] fp16 block (128B swizzle)

// ---------------------------------------------------------------------------
// host: tensor maps
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// 3D map over a [BH][L][cols] tensor, box [1][128][box_cols], 128B swizzle.
int make_map(CUtensorMap *m, const void *base, CUtensorMapDataType type, int esize, int BH, int L,
             int cols, int box_cols) {
    auto enc = encoder();
    if (!enc) return FAVOR_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)L, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)cols * esize, (cuuint64_t)L * cols * esize};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, type, 3, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FAVOR_OK : FAVOR_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
struct Geo {
    int d, dv, r, nproj, map, n_ft, np_tile;   // np_tile: projections per 128-feature tile
};

__device__ __forceinline__ uint32_t tm_addr(uint32_t base, int quarter, int col) {
    return base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col;
}

__device__ __forceinline__ void set_status(int *status, int code) {
    if (status) atomicExch(status, code);
}

// warp + CTA reductions over kThreads threads; `red` holds 8 floats.
__device__ __forceinline__ float cta_max(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < kThreads / 32; ++i) r = fmaxf(r, red[i]);
    return r;
}

__device__ __forceinline__ float cta_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = 0.f;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) r += red[i];
    return r;
}

// In-place bf16 -> fp16 conversion of a [128][64*nblk] tile (128B-swizzled
// blocks of 16 KB).  Thread (row = tid % 128, half = tid / 128) converts four
// 16-byte chunks of its row per block, rotating the chunk index with the row
// so that eight consecutive rows hit distinct banks.  Returns this thread's
// partial sum of squares and max |x| over its chunks.
__device__ __forceinline__ void convert_tile(uint8_t *tile, int nblk, float &sumsq, float &amax) {
    const int row = threadIdx.x & 127, half = threadIdx.x >> 7;
    sumsq = 0.f;
    amax = 0.f;
    for (int b = 0; b < nblk; ++b) {
        uint8_t *rp = tile + b * kBlk + row * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            int p = (half * 4 + c + row) & 7;
            uint4 *ptr = reinterpret_cast<uint4 *>(rp + p * 16);
            uint4 u = *ptr;
            uint32_t w[4] = {u.x, u.y, u.z, u.w}, o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
                sumsq = fmaf(lo, lo, fmaf(hi, hi, sumsq));
                amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
                o[i] = pack_half2(lo, hi);
            }
            *ptr = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// Store 32 features (fp16) of one row into a 128B-swizzled [128][64] block at
// columns [c0, c0 + 32).
__device__ __forceinline__ void store_row32(uint8_t *blk, int row, int c0, const float (&v)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 u = make_uint4(pack_half2(v[8 * c + 0], v[8 * c + 1]), pack_half2(v[8 * c + 2], v[8 * c + 3]),
                             pack_half2(v[8 * c + 4], v[8 * c + 5]), pack_half2(v[8 * c + 6], v[8 * c + 7]));
        *reinterpret_cast<uint4 *>(blk + sw128_offset(row, c0 + 8 * c)) = u;
    }
}

__device__ __forceinline__ float half_lo(uint32_t u) { return __half2float(__ushort_as_half((unsigned short)(u & 0xffff))); }
__device__ __forceinline__ float half_hi(uint32_t u) { return __half2float(__ushort_as_half((unsigned short)(u >> 16))); }

// Reload 32 fp16 features of a row (as stored by store_row32) into floats.
__device__ __forceinline__ void load_row32(const uint8_t *blk, int row, int c0, float (&v)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 u = *reinterpret_cast<const uint4 *>(blk + sw128_offset(row, c0 + 8 * c));
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[8 * c + 2 * i] = half_lo(w[i]);
            v[8 * c + 2 * i + 1] = half_hi(w[i]);
        }
    }
}

// sin/cos with the argument first reduced to [-pi, pi] (Cody-Waite, 2pi split
// in three parts) so that the hardware approximations stay accurate for
// projections of any size met here.
__device__ __forceinline__ void sincos_reduced(float x, float &s, float &c) {
    const float inv2pi = 0.15915494309189535f;
    const float p1 = 6.28125f, p2 = 1.9353071795864769e-3f, p3 = 0.0f;
    float n = rintf(x * inv2pi);
    float t = fmaf(-n, p1, x);
    t = fmaf(-n, p2, t);
    t = fmaf(-n, p3, t);
    __sincosf(t, &s, &c);
}

// ELU + 1 ("Kernel Feature Maps" section 1); p is x itself here.
__device__ __forceinline__ float elu1(float p) { return p > 0.f ? p + 1.f : ex2(p * kLog2e); }

// ---------------------------------------------------------------------------
// W image: fp16, 128B-swizzled K-major blocks [nproj][64] per 64 columns of d,
// scaled by log2(e) for the positive map; the identity for elu1.
// ---------------------------------------------------------------------------
__global__ void tc_prep_omega(const float *__restrict__ omega, uint8_t *__restrict__ img, int H,
                              int nproj, int d, int map) {
    const int h = blockIdx.y;
    const size_t per = (size_t)nproj * d;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < per;
         e += (size_t)gridDim.x * blockDim.x) {
        int p = (int)(e / d), j = (int)(e % d);
        float w;
        if (map == FAVOR_MAP_ELU1) w = (p == j) ? 1.f : 0.f;
        else w = omega[(size_t)h * per + e] * (map == FAVOR_MAP_POSITIVE ? kLog2e : 1.f);
        uint8_t *blk = img + (size_t)h * per * 2 + (size_t)(j / 64) * nproj * 128;
        *reinterpret_cast<__half *>(blk + sw128_offset(p, j % 64)) = __float2half_rn(w);
    }
}

// ---------------------------------------------------------------------------
// Key feature epilogue (shared by tc_state and tc_causal).
// P (projections) for n_tiles feature tiles sits in TMEM columns [128 t, ...).
// Writes fp16 key features for tokens < valid into phk (K-major blocks of 64
// features, two per tile), zeros for the rest.  Positive map: updates the
// key reference *R (log2 units) when this chunk exceeds it; returns the
// factor alpha = 2^(R_old - R_new) the existing state must be scaled by (1
// if unchanged) and the chunk's key mass (sum over tokens of the largest
// feature) in *mass.
// ---------------------------------------------------------------------------
struct KeyEpi {
    float *R;        // smem scalar
    float *nk;       // [128] |k|^2 log2e / 2
    float *part;     // [2][128] half-row partials
    float *red;      // [8]
};

__device__ float key_features(const Geo &g, uint32_t tmem, int first_tile, int n_tiles,
                              uint8_t *phk, int valid, const KeyEpi &ep, float *mass) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, h = warp >> 2;
    const int row = q * 32 + lane;
    const bool ok = row < valid;
    float alpha = 1.f;
    float mf = 0.f;   // largest feature of this row (this thread's columns)
    if (g.map == FAVOR_MAP_POSITIVE) {
        // pass 1: row maximum of w.k (log2 units)
        float mx = -INFINITY;
        for (int t = 0; t < n_tiles; ++t) {
            for (int c = 0; c < 2; ++c) {
                float v[32];
                tmem_ld32(tm_addr(tmem, q, 128 * (first_tile + t) + 64 * h + 32 * c), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) mx = fmaxf(mx, v[i]);
            }
        }
        float lam = ok ? mx - ep.nk[row] : -INFINITY;
        float mu = cta_max(lam, ep.red);
        float Rold = *ep.R;
        float Rnew = Rold;
        if (mu > -INFINITY && (Rold == -INFINITY || mu > Rold + kShift + kSlack)) Rnew = mu - kShift;
        __syncthreads();
        if (threadIdx.x == 0) *ep.R = Rnew;
        alpha = (Rold == -INFINITY) ? 0.f : ex2(Rold - Rnew);
        const float off = (ok ? ep.nk[row] : 0.f) + Rnew;
        // pass 2: features
        for (int t = 0; t < n_tiles; ++t) {
            uint8_t *blk = phk + (size_t)(2 * t + h) * kBlk;
            for (int c = 0; c < 2; ++c) {
                float v[32];
                tmem_ld32(tm_addr(tmem, q, 128 * (first_tile + t) + 64 * h + 32 * c), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v[i] = ok ? ex2(v[i] - off) : 0.f;
                    mf = fmaxf(mf, v[i]);
                }
                store_row32(blk, row, 32 * c, v);
            }
        }
    } else if (g.map == FAVOR_MAP_TRIG) {
        // projection tile t holds 64 columns: sin -> block 2t, cos -> block 2t+1
        for (int t = 0; t < n_tiles; ++t) {
            float v[32], s[32], co[32];
            tmem_ld32(tm_addr(tmem, q, 128 * (first_tile + t) + 32 * h), v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (ok) sincos_reduced(v[i], s[i], co[i]);
                else s[i] = co[i] = 0.f;
                mf = fmaxf(mf, fmaxf(fabsf(s[i]), fabsf(co[i])));
            }
            store_row32(phk + (size_t)(2 * t) * kBlk, row, 32 * h, s);
            store_row32(phk + (size_t)(2 * t + 1) * kBlk, row, 32 * h, co);
        }
    } else {
        for (int t = 0; t < n_tiles; ++t) {
            uint8_t *blk = phk + (size_t)(2 * t + h) * kBlk;
            for (int c = 0; c < 2; ++c) {
                float v[32];
                tmem_ld32(tm_addr(tmem, q, 128 * (first_tile + t) + 64 * h + 32 * c), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v[i] = ok ? elu1(v[i]) : 0.f;
                    mf = fmaxf(mf, v[i]);
                }
                store_row32(blk, row, 32 * c, v);
            }
        }
    }
    // per-row largest feature (combine the two column halves), then the chunk mass
    ep.part[h * 128 + row] = mf;
    __syncthreads();
    float rowmax = fmaxf(ep.part[row], ep.part[128 + row]);
    float m = cta_sum(h == 0 ? rowmax : 0.f, ep.red);
    *mass = m;
    return alpha;
}

// Convert a key tile in place and publish |k|^2 log2e / 2 per row.
__device__ void key_tile_prepare(uint8_t *xk, int nd, float *nk, float *part) {
    float ss, am;
    convert_tile(xk, nd, ss, am);
    const int row = threadIdx.x & 127, half = threadIdx.x >> 7;
    part[half * 128 + row] = ss;
    __syncthreads();
    if (half == 0) nk[row] = 0.5f * kLog2e * (part[row] + part[128 + row]);
}

// ---------------------------------------------------------------------------
// MMA issue helpers (one thread)
// ---------------------------------------------------------------------------
// P[:, 128 t .. ] = X W_tile^T for feature tiles [t0, t0 + nt); X K-major
// [128][d] in nd blocks; W image K-major [nproj][64] per d block.
// W image in smem: K-major blocks of w_rows rows per 64 columns of d.
__device__ __forceinline__ void issue_projection(const Geo &g, uint32_t tmem, uint32_t x_s,
                                                 uint32_t w_s, int w_rows, int t0, int nt, int col0) {
    const uint32_t idesc = idesc_f16(128, g.np_tile, 0, 0);
    const int nk = g.d / 16;
    for (int t = 0; t < nt; ++t) {
        const int p0 = (t0 + t) * g.np_tile;
        for (int kk = 0; kk < nk; ++kk) {
            uint64_t a = smem_desc(x_s + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
            uint64_t b = smem_desc(w_s + (kk >> 2) * (uint32_t)w_rows * 128 + p0 * 128 + (kk & 3) * 32,
                                   16, 1024);
            mma_f16(tmem + col0 + 128 * t, a, b, idesc, kk > 0);
        }
    }
}

// S_tile[t] (M = 128 features, N = 64 values) += phi_K^T V and z += phi_K^T 1,
// for feature tiles t in [0, nt); phk blocks (2t, 2t+1) are the MN-major A
// operand; V (MN-major, one 64-wide block) and the ones block (K-major [16][128]).
__device__ __forceinline__ void issue_state_update(uint32_t tmem, uint32_t phk_s, uint32_t v_s,
                                                   uint32_t ones_s, int nt, int col_s,
                                                   int stride_cols, int nvblk) {
    for (int t = 0; t < nt; ++t) {
        for (int vb = 0; vb < nvblk; ++vb) {
            const uint32_t idesc = idesc_f16(128, 64, 1, 1);
            for (int kk = 0; kk < kC / 16; ++kk) {
                uint64_t a = smem_desc(phk_s + (2 * t) * kBlk + kk * 2048, kBlk, 1024);
                uint64_t b = smem_desc(v_s + vb * kBlk + kk * 2048, kBlk, 1024);
                mma_f16(tmem + col_s + t * stride_cols + 64 * vb, a, b, idesc, 1);
            }
        }
        const uint32_t idz = idesc_f16(128, 16, 1, 0);
        for (int kk = 0; kk < kC / 16; ++kk) {
            uint64_t a = smem_desc(phk_s + (2 * t) * kBlk + kk * 2048, kBlk, 1024);
            uint64_t b = smem_desc(ones_s + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024);
            mma_f16(tmem + col_s + t * stride_cols + 64 * nvblk, a, b, idz, 1);
        }
    }
}

// ---------------------------------------------------------------------------
// tc_state: per (feature tile, segment, head) the segment state
//   S[f][c] = sum_t phi(k_t)_f v_t[c],  z[f] = sum_t phi(k_t)_f
// at key reference R, written as fp32 [f][dv + 1] plus (R, mass, vmax).
// ---------------------------------------------------------------------------
struct StateArgs {
    Geo g;
    int H, L, seg_len, nseg;
    const uint8_t *omg;       // [H] images
    float *state;             // [BH][nseg][r][dv+1]
    float *meta;              // [BH][nseg][n_ft][4]: R, mass, vmax, -
    int *status;
    uint32_t o_w, o_xk, o_xv, o_phk, o_ones, o_small, tmem_cols;
};

__global__ void __launch_bounds__(kThreads, 1)
tc_state(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
         const StateArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Geo &g = a.g;
    const int ft = blockIdx.x, seg = blockIdx.y, bh = blockIdx.z, head = bh % a.H;
    const int t_begin = seg * a.seg_len, t_end = min(a.L, t_begin + a.seg_len);
    const int nchunk = (t_end - t_begin + kC - 1) / kC;
    const int nd = g.d / 64, nvb = g.dv / 64;
    uint8_t *w = sm + a.o_w, *xk = sm + a.o_xk, *xv = sm + a.o_xv, *phk = sm + a.o_phk,
            *ones = sm + a.o_ones;
    float *small = reinterpret_cast<float *>(sm + a.o_small);
    float *nk = small, *part = small + 128, *red = small + 384, *Rp = small + 392;
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + 400);   // 0: w, 1: k, 2: v, 3: mma
    uint32_t *tslot = reinterpret_cast<uint32_t *>(small + 408);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3, h = warp >> 2;

    // ones block for the z column
    for (int i = threadIdx.x; i < 4096 / 16; i += kThreads)
        reinterpret_cast<uint4 *>(ones)[i] = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        *Rp = -INFINITY;
    }
    if (warp == 0) tmem_alloc(tslot, a.tmem_cols);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int col_s = 128;                   // S at [128, 128 + dv), z at [128 + dv, +16)
    uint32_t ph_k = 0, ph_v = 0, ph_m = 0;
    bool alive = true;

    if (threadIdx.x == 0) {
        // W rows of this feature tile: np_tile rows per d block
        const uint32_t wbytes = (uint32_t)g.np_tile * 128;
        mbar_arrive_expect_tx(&bars[0], wbytes * nd);
        for (int b = 0; b < nd; ++b)
            bulk_load(w + b * wbytes, a.omg + (size_t)head * g.nproj * g.d * 2 +
                                          (size_t)b * g.nproj * 128 + (size_t)ft * wbytes,
                      wbytes, &bars[0]);
        if (nchunk > 0) {
            mbar_arrive_expect_tx(&bars[1], kBlk * nd);
            for (int b = 0; b < nd; ++b) tma_load_3d(xk + b * kBlk, &tm_k, &bars[1], 64 * b, t_begin, bh);
            mbar_arrive_expect_tx(&bars[2], kBlk * nvb);
            for (int b = 0; b < nvb; ++b) tma_load_3d(xv + b * kBlk, &tm_v, &bars[2], 64 * b, t_begin, bh);
        }
    }
    // zero S and z
    {
        float zero[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) zero[i] = 0.f;
        for (int c = 32 * h; c < g.dv + 16; c += 64) tmem_st32(tm_addr(tmem, q, col_s + c), zero);
        tmem_st_wait();
    }
    alive = mbar_wait(&bars[0], 0, kWaitLimit);
    float mass_total = 0.f, vmax = 0.f;
    const uint32_t w_s = smem_u32(w), xk_s = smem_u32(xk), xv_s = smem_u32(xv),
                   phk_s = smem_u32(phk), ones_s = smem_u32(ones);
    KeyEpi ep{Rp, nk, part, red};

    for (int c = 0; c < nchunk; ++c) {
        const int tc0 = t_begin + c * kC;
        const int valid = min(kC, t_end - tc0);
        alive = alive && mbar_wait(&bars[1], ph_k, kWaitLimit);
        ph_k ^= 1;
        if (__syncthreads_or(!alive)) break;
        key_tile_prepare(xk, nd, nk, part);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (threadIdx.x == 0) {
            issue_projection(g, tmem, xk_s, w_s, g.np_tile, 0, 1, 0);
            mma_commit(&bars[3]);
        }
        alive = mbar_wait(&bars[3], ph_m, kWaitLimit);
        ph_m ^= 1;
        if (__syncthreads_or(!alive)) break;
        tc_fence_after();
        // the K tile is free: prefetch the next one
        if (threadIdx.x == 0 && c + 1 < nchunk) {
            mbar_arrive_expect_tx(&bars[1], kBlk * nd);
            for (int b = 0; b < nd; ++b) tma_load_3d(xk + b * kBlk, &tm_k, &bars[1], 64 * b, tc0 + kC, bh);
        }
        float mass;
        float alpha = key_features(g, tmem, 0, 1, phk, valid, ep, &mass);
        if (alpha != 1.f) {
            // rescale the running state to the new reference
            for (int cc = 32 * h; cc < g.dv + 16; cc += 64) {
                float v[32];
                tmem_ld32(tm_addr(tmem, q, col_s + cc), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= alpha;
                tmem_st32(tm_addr(tmem, q, col_s + cc), v);
            }
            tmem_st_wait();
            mass_total *= alpha;
        }
        mass_total += mass;
        alive = alive && mbar_wait(&bars[2], ph_v, kWaitLimit);
        ph_v ^= 1;
        if (__syncthreads_or(!alive)) break;
        float ss, am;
        convert_tile(xv, nvb, ss, am);
        vmax = fmaxf(vmax, cta_max(am, red));
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (threadIdx.x == 0) {
            issue_state_update(tmem, phk_s, xv_s, ones_s, 1, col_s, 0, nvb);
            mma_commit(&bars[3]);
        }
        alive = mbar_wait(&bars[3], ph_m, kWaitLimit);
        ph_m ^= 1;
        if (__syncthreads_or(!alive)) break;
        tc_fence_after();
        if (threadIdx.x == 0 && c + 1 < nchunk) {
            mbar_arrive_expect_tx(&bars[2], kBlk * nvb);
            for (int b = 0; b < nvb; ++b) tma_load_3d(xv + b * kBlk, &tm_v, &bars[2], 64 * b, tc0 + kC, bh);
        }
    }
    if (alive) {
        // S, z -> global: thread (q, lane) owns feature ft*128 + 32q + lane; halves split columns
        const int f = ft * 128 + q * 32 + lane;
        float *dst = a.state + (((size_t)bh * a.nseg + seg) * g.r + f) * (g.dv + 1);
        for (int cc = 32 * h; cc < g.dv; cc += 64) {
            float v[32];
            tmem_ld32(tm_addr(tmem, q, col_s + cc), v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[cc + i] = v[i];
        }
        if (h == 0) {
            float v[16];
            tmem_ld16(tm_addr(tmem, q, col_s + g.dv), v);
            tmem_ld_wait();
            dst[g.dv] = v[0];
        }
        if (threadIdx.x == 0) {
            float *m = a.meta + (((size_t)bh * a.nseg + seg) * g.n_ft + ft) * 4;
            m[0] = *Rp;
            m[1] = mass_total;
            m[2] = vmax;
            m[3] = 0.f;
        }
    } else {
        set_status(a.status, FAVOR_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, a.tmem_cols);
}

// ---------------------------------------------------------------------------
// tc_combine: fixed-order combination of segment states.
//  non-causal (one block per head): KV = sum_g S_g 2^(R_g - R*), z likewise;
//    sigma = power of two with max|sigma KV| <= 16384; writes the fp16 state
//    operand image [nvb][r][64] (128B-swizzled MN-major), z (fp32), sigma.
//  causal (block per head and segment s >= 1): S_in(s) = sum_{g<s} ..., fp32
//    [r][dv+1], plus (R_in, max_f z_f, vmax_in).
// ---------------------------------------------------------------------------
struct CombineArgs {
    Geo g;
    int nseg;              // segment states available
    int causal;
    const float *state, *meta;
    uint8_t *sop;          // non-causal: [BH][nvb][r][64] fp16 image
    float *zout;           // non-causal: [BH][r]
    float *sig;            // non-causal: [BH]
    float *s_in;           // causal: [BH][nseg+1][r][dv+1]
    float *meta_in;        // causal: [BH][nseg+1][4]
};

__global__ void tc_combine(const CombineArgs a) {
    const Geo &g = a.g;
    const int bh = blockIdx.x;
    const int upto = a.causal ? blockIdx.y + 1 : a.nseg;   // segments [0, upto)
    __shared__ float red[32];
    __shared__ float sh_R;
    const float *meta = a.meta + (size_t)bh * a.nseg * g.n_ft * 4;
    // reference: max over segments and feature tiles
    float R = -INFINITY;
    for (int i = threadIdx.x; i < upto * g.n_ft; i += blockDim.x) R = fmaxf(R, meta[i * 4]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) R = fmaxf(R, __shfl_xor_sync(0xffffffffu, R, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = R;
    __syncthreads();
    if (threadIdx.x == 0) {
        float r = -INFINITY;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r = fmaxf(r, red[i]);
        sh_R = r;
    }
    __syncthreads();
    R = sh_R;
    __syncthreads();
    const int W = g.dv + 1;
    const size_t per = (size_t)g.r * W;
    const float *st = a.state + (size_t)bh * a.nseg * per;
    float amax = 0.f, zmax = 0.f, vmax = 0.f;
    // pass 1: sums into the output buffer (causal) or registers-free second pass (non-causal)
    float *dst = a.causal ? a.s_in + ((size_t)bh * (a.nseg + 1) + upto) * per : nullptr;
    for (size_t e = threadIdx.x; e < per; e += blockDim.x) {
        const int f = (int)(e / W), c = (int)(e % W);
        const int ftile = f / 128;
        float s = 0.f;
        for (int gi = 0; gi < upto; ++gi) {
            float Rg = meta[(gi * g.n_ft + ftile) * 4];
            float sc = (Rg == -INFINITY || R == -INFINITY) ? 0.f : ex2(Rg - R);
            if (g.map != FAVOR_MAP_POSITIVE) sc = 1.f;
            s += st[gi * per + e] * sc;
        }
        if (c < g.dv) amax = fmaxf(amax, fabsf(s));
        else zmax = fmaxf(zmax, fabsf(s));
        if (a.causal) {
            dst[e] = s;
        } else if (c == g.dv) {
            a.zout[(size_t)bh * g.r + f] = s;
        }
    }
    for (int gi = threadIdx.x; gi < upto * g.n_ft; gi += blockDim.x) vmax = fmaxf(vmax, meta[gi * 4 + 2]);
    // block maxima
    float vals[3] = {amax, zmax, vmax};
    for (int k = 0; k < 3; ++k) {
        float v = vals[k];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        __syncthreads();
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
        __syncthreads();
        float r = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r = fmaxf(r, red[i]);
        vals[k] = r;
    }
    if (a.causal) {
        if (threadIdx.x == 0) {
            float *m = a.meta_in + ((size_t)bh * (a.nseg + 1) + upto) * 4;
            m[0] = (g.map == FAVOR_MAP_POSITIVE) ? R : 0.f;
            m[1] = vals[1];
            m[2] = vals[2];
            m[3] = 0.f;
        }
        return;
    }
    // non-causal: sigma and the fp16 operand image (second pass over the sums)
    float sigma = 1.f;
    if (vals[0] > 0.f) sigma = exp2f(floorf(log2f(kSigmaTarget / vals[0])));
    if (threadIdx.x == 0) a.sig[bh] = sigma;
    const int nvb = g.dv / 64;
    uint8_t *img = a.sop + (size_t)bh * nvb * g.r * 128;
    for (size_t e = threadIdx.x; e < (size_t)g.r * g.dv; e += blockDim.x) {
        const int f = (int)(e / g.dv), c = (int)(e % g.dv);
        const int ftile = f / 128;
        float s = 0.f;
        for (int gi = 0; gi < upto; ++gi) {
            float Rg = meta[(gi * g.n_ft + ftile) * 4];
            float sc = (Rg == -INFINITY || R == -INFINITY) ? 0.f : ex2(Rg - R);
            if (g.map != FAVOR_MAP_POSITIVE) sc = 1.f;
            s += st[gi * per + (size_t)f * W + c] * sc;
        }
        *reinterpret_cast<__half *>(img + (size_t)(c / 64) * g.r * 128 + sw128_offset(f, c % 64)) =
            __float2half_rn(s * sigma);
    }
}

// ---------------------------------------------------------------------------
// Query feature epilogue (tc_output, tc_causal).  P for all n_ft tiles is in
// TMEM [0, 128 n_ft).  Writes fp16 query features to phq (blocks of 64) and
// returns this thread's partial phi(q) . z over its columns (z fp32 in smem).
// ---------------------------------------------------------------------------
__device__ float query_features(const Geo &g, uint32_t tmem, uint8_t *phq, const float *zs,
                                float *part) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, h = warp >> 2;
    const int row = q * 32 + lane;
    float den = 0.f;
    if (g.map == FAVOR_MAP_POSITIVE) {
        float mx = -INFINITY;
        for (int t = 0; t < g.n_ft; ++t)
            for (int c = 0; c < 2; ++c) {
                float v[32];
                tmem_ld32(tm_addr(tmem, q, 128 * t + 64 * h + 32 * c), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) mx = fmaxf(mx, v[i]);
            }
        part[h * 128 + row] = mx;
        __syncthreads();
        const float off = fmaxf(part[row], part[128 + row]) - kShift;
        for (int t = 0; t < g.n_ft; ++t) {
            uint8_t *blk = phq + (size_t)(2 * t + h) * kBlk;
            for (int c = 0; c < 2; ++c) {
                float v[32];
                tmem_ld32(tm_addr(tmem, q, 128 * t + 64 * h + 32 * c), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = ex2(v[i] - off);
                store_row32(blk, row, 32 * c, v);
                float r[32];
                load_row32(blk, row, 32 * c, r);   // the rounded values the MMA sees
                const float *z = zs + 128 * t + 64 * h + 32 * c;
#pragma unroll
                for (int i = 0; i < 32; ++i) den = fmaf(r[i], z[i], den);
            }
        }
    } else if (g.map == FAVOR_MAP_TRIG) {
        for (int t = 0; t < g.n_ft; ++t) {
            float v[32], s[32], co[32];
            tmem_ld32(tm_addr(tmem, q, 128 * t + 32 * h), v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) sincos_reduced(v[i], s[i], co[i]);
            uint8_t *bs = phq + (size_t)(2 * t) * kBlk, *bc = phq + (size_t)(2 * t + 1) * kBlk;
            store_row32(bs, row, 32 * h, s);
            store_row32(bc, row, 32 * h, co);
            float rs[32], rc[32];
            load_row32(bs, row, 32 * h, rs);
            load_row32(bc, row, 32 * h, rc);
            const float *zsn = zs + 128 * t + 32 * h, *zco = zs + 128 * t + 64 + 32 * h;
#pragma unroll
            for (int i = 0; i < 32; ++i) den = fmaf(rs[i], zsn[i], fmaf(rc[i], zco[i], den));
        }
    } else {
        for (int t = 0; t < g.n_ft; ++t) {
            uint8_t *blk = phq + (size_t)(2 * t + h) * kBlk;
            for (int c = 0; c < 2; ++c) {
                float v[32];
                tmem_ld32(tm_addr(tmem, q, 128 * t + 64 * h + 32 * c), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = elu1(v[i]);
                store_row32(blk, row, 32 * c, v);
                float r[32];
                load_row32(blk, row, 32 * c, r);
                const float *z = zs + 128 * t + 64 * h + 32 * c;
#pragma unroll
                for (int i = 0; i < 32; ++i) den = fmaf(r[i], z[i], den);
            }
        }
    }
    return den;
}

// D (M = 128 queries, N = 64) = phi_Q S_op over K = r features.
__device__ __forceinline__ void issue_inter(const Geo &g, uint32_t tmem_d, uint32_t phq_s,
                                            uint32_t sop_s, int accumulate_first) {
    const uint32_t idesc = idesc_f16(128, 64, 0, 1);
    for (int kk = 0; kk < g.r / 16; ++kk) {
        uint64_t a = smem_desc(phq_s + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
        uint64_t b = smem_desc(sop_s + kk * 2048, kBlk, 1024);
        mma_f16(tmem_d, a, b, idesc, (kk > 0) || accumulate_first);
    }
}

// Write a [128][64] fp32 output tile (values given per thread: row, 32
// columns at 32 h) into the staging area as two 128B-swizzled [128][32]
// halves for the TMA store.
__device__ __forceinline__ void stage_out(uint8_t *stage, int row, int h, const float (&o)[32]) {
    uint8_t *half = stage + h * kBlk;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        int p = (c ^ (row & 7));
        *reinterpret_cast<float4 *>(half + row * 128 + p * 16) =
            make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
    }
}

// ---------------------------------------------------------------------------
// tc_output: non-causal rows.  Grid (row groups, dv tiles, heads).
// ---------------------------------------------------------------------------
struct OutputArgs {
    Geo g;
    int H, L, chunks_per_cta;
    const uint8_t *omg, *sop;
    const float *z, *sig;
    int *status;
    uint32_t o_w, o_xq, o_sop, o_phq, o_stage, o_small, tmem_cols;
};

__global__ void __launch_bounds__(kThreads, 1)
tc_output(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_out,
          const OutputArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Geo &g = a.g;
    const int dvt = blockIdx.y, bh = blockIdx.z, head = bh % a.H;
    const int nchunk_total = (a.L + kC - 1) / kC;
    const int c_begin = blockIdx.x * a.chunks_per_cta;
    const int c_end = min(nchunk_total, c_begin + a.chunks_per_cta);
    const int nd = g.d / 64;
    uint8_t *w = sm + a.o_w, *xq = sm + a.o_xq, *sop = sm + a.o_sop, *phq = sm + a.o_phq,
            *stage = sm + a.o_stage;
    float *small = reinterpret_cast<float *>(sm + a.o_small);
    float *zs = small, *part = small + 256, *dpart = small + 512;
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + 776);   // 0: w+sop, 1: q, 2: mma
    uint32_t *tslot = reinterpret_cast<uint32_t *>(small + 784);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3, h = warp >> 2;
    const int row = q * 32 + lane;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, a.tmem_cols);
    for (int f = threadIdx.x; f < g.r; f += kThreads) zs[f] = a.z[(size_t)bh * g.r + f];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int col_d = 256;
    const float inv_sigma = 1.f / a.sig[bh];
    if (threadIdx.x == 0 && c_begin < c_end) {
        const uint32_t wbytes = (uint32_t)g.nproj * g.d * 2, sbytes = (uint32_t)g.r * 128;
        mbar_arrive_expect_tx(&bars[0], wbytes + sbytes);
        bulk_load(w, a.omg + (size_t)head * wbytes, wbytes, &bars[0]);
        bulk_load(sop, a.sop + ((size_t)bh * (g.dv / 64) + dvt) * sbytes, sbytes, &bars[0]);
        mbar_arrive_expect_tx(&bars[1], kBlk * nd);
        for (int b = 0; b < nd; ++b) tma_load_3d(xq + b * kBlk, &tm_q, &bars[1], 64 * b, c_begin * kC, bh);
    }
    bool alive = mbar_wait(&bars[0], 0, kWaitLimit);
    uint32_t ph_q = 0, ph_m = 0;
    const uint32_t w_s = smem_u32(w), xq_s = smem_u32(xq), sop_s = smem_u32(sop), phq_s = smem_u32(phq);
    for (int c = c_begin; c < c_end; ++c) {
        alive = alive && mbar_wait(&bars[1], ph_q, kWaitLimit);
        ph_q ^= 1;
        if (__syncthreads_or(!alive)) break;
        float ss, am;
        convert_tile(xq, nd, ss, am);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (threadIdx.x == 0) {
            issue_projection(g, tmem, xq_s, w_s, g.nproj, 0, g.n_ft, 0);
            mma_commit(&bars[2]);
        }
        alive = mbar_wait(&bars[2], ph_m, kWaitLimit);
        ph_m ^= 1;
        if (__syncthreads_or(!alive)) break;
        tc_fence_after();
        if (threadIdx.x == 0 && c + 1 < c_end) {
            mbar_arrive_expect_tx(&bars[1], kBlk * nd);
            for (int b = 0; b < nd; ++b) tma_load_3d(xq + b * kBlk, &tm_q, &bars[1], 64 * b, (c + 1) * kC, bh);
        }
        float den = query_features(g, tmem, phq, zs, part);
        dpart[h * 128 + row] = den;
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (threadIdx.x == 0) {
            issue_inter(g, tmem + col_d, phq_s, sop_s, 0);
            mma_commit(&bars[2]);
        }
        alive = mbar_wait(&bars[2], ph_m, kWaitLimit);
        ph_m ^= 1;
        if (__syncthreads_or(!alive)) break;
        tc_fence_after();
        const float dn = dpart[row] + dpart[128 + row];
        float o[32];
        tmem_ld32(tm_addr(tmem, q, col_d + 32 * h), o);
        tmem_ld_wait();
        const float scale = inv_sigma / dn;
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= scale;
        if (threadIdx.x == 0) bulk_wait_read0();
        __syncthreads();
        stage_out(stage, row, h, o);
        fence_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            tma_store_3d(&tm_out, stage, 64 * dvt, c * kC, bh);
            tma_store_3d(&tm_out, stage + kBlk, 64 * dvt + 32, c * kC, bh);
            bulk_commit();
        }
    }
    if (threadIdx.x == 0) bulk_wait0();
    if (!alive) set_status(a.status, FAVOR_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, a.tmem_cols);
}

// ---------------------------------------------------------------------------
// tc_causal: the chunked causal scan.  Grid (segments, dv tiles, heads).
// TMEM columns: P / A [0, 256), A V at [128, 192), phi_Q S at [256, 320),
// state tiles [320 + 96 t, ...): 64 values, then z (the MMA writes 16 copies
// of z; the slot keeps 32 columns so 32-wide loads and stores stay inside it).
// ---------------------------------------------------------------------------
struct CausalArgs {
    Geo g;
    int H, L, seg_len, nseg;
    const uint8_t *omg;
    const float *s_in, *meta_in;   // [BH][nseg][r][dv+1], [BH][nseg][4] (segment 0 unused)
    int *status;
    uint32_t o_w, o_xq, o_xk, o_xv, o_phq, o_phk, o_ones, o_small, tmem_cols;
};

__global__ void __launch_bounds__(kThreads, 1)
tc_causal(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
          const CausalArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Geo &g = a.g;
    const int seg = blockIdx.x, dvt = blockIdx.y, bh = blockIdx.z, head = bh % a.H;
    const int t_begin = seg * a.seg_len, t_end = min(a.L, t_begin + a.seg_len);
    const int nchunk = (t_end - t_begin + kC - 1) / kC;
    const int nd = g.d / 64, nft = g.n_ft;
    uint8_t *w = sm + a.o_w, *xq = sm + a.o_xq, *xk = sm + a.o_xk, *xv = sm + a.o_xv,
            *phq = sm + a.o_phq, *phk = sm + a.o_phk, *ones = sm + a.o_ones;
    uint8_t *sop = xq;      // state operand [r][64] fp16 (aliases the Q and K tiles)
    uint8_t *bhat = phq;    // normalised intra-chunk matrix (aliases phi_Q)
    uint8_t *stage = phk;   // output staging (aliases phi_K)
    float *small = reinterpret_cast<float *>(sm + a.o_small);
    float *zs = small;                  // [256]
    float *nk = small + 256;            // [128]
    float *part = small + 384;          // [256]
    float *dpart = small + 640;         // [256] den_inter partials
    float *rho = small + 896;           // [128]
    float *deni = small + 1024;         // [128]
    float *red = small + 1152;          // [8]
    float *sc = small + 1160;           // scalars: 0 R, 1 zmax, 2 vmax, 3 alpha_pending
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + 1168);   // 0 w, 1 qk, 2 v, 3 mma
    uint32_t *tslot = reinterpret_cast<uint32_t *>(small + 1184);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3, h = warp >> 2;
    const int row = q * 32 + lane;
    const int col_a = 0, col_da = 128, col_di = 256, col_s = 320, s_stride = 96;

    for (int i = threadIdx.x; i < 4096 / 16; i += kThreads)
        reinterpret_cast<uint4 *>(ones)[i] = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        const float *m = a.meta_in + ((size_t)bh * a.nseg + seg) * 4;
        const bool has_in = seg > 0;
        sc[0] = has_in ? m[0] : (g.map == FAVOR_MAP_POSITIVE ? -INFINITY : 0.f);
        sc[1] = has_in ? m[1] : 0.f;
        sc[2] = has_in ? m[2] : 0.f;
        sc[3] = 1.f;
    }
    if (warp == 0) tmem_alloc(tslot, a.tmem_cols);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (threadIdx.x == 0) {
        const uint32_t wbytes = (uint32_t)g.nproj * g.d * 2;
        mbar_arrive_expect_tx(&bars[0], wbytes);
        bulk_load(w, a.omg + (size_t)head * wbytes, wbytes, &bars[0]);
        if (nchunk > 0) {
            mbar_arrive_expect_tx(&bars[1], 2 * kBlk * nd);
            for (int b = 0; b < nd; ++b) {
                tma_load_3d(xq + b * kBlk, &tm_q, &bars[1], 64 * b, t_begin, bh);
                tma_load_3d(xk + b * kBlk, &tm_k, &bars[1], 64 * b, t_begin, bh);
            }
            mbar_arrive_expect_tx(&bars[2], kBlk);
            tma_load_3d(xv, &tm_v, &bars[2], 64 * dvt, t_begin, bh);
        }
    }
    // initial state: S_in of this segment (or zero) -> TMEM state tiles
    for (int t = 0; t < nft; ++t) {
        const int f = t * 128 + row;
        const float *src = (seg > 0) ? a.s_in + (((size_t)bh * a.nseg + seg) * g.r + f) * (g.dv + 1) : nullptr;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = src ? src[64 * dvt + 32 * h + i] : 0.f;
        tmem_st32(tm_addr(tmem, q, col_s + t * s_stride + 32 * h), v);
        if (h == 0) {
            const float zval = src ? src[g.dv] : 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = zval;
            tmem_st32(tm_addr(tmem, q, col_s + t * s_stride + 64), v);
        }
    }
    tmem_st_wait();
    bool alive = mbar_wait(&bars[0], 0, kWaitLimit);
    uint32_t ph_qk = 0, ph_v = 0, ph_m = 0;
    const uint32_t w_s = smem_u32(w), xq_s = smem_u32(xq), xk_s = smem_u32(xk), xv_s = smem_u32(xv),
                   phq_s = smem_u32(phq), phk_s = smem_u32(phk), ones_s = smem_u32(ones),
                   sop_s = smem_u32(sop), bhat_s = smem_u32(bhat);
    KeyEpi ep{&sc[0], nk, part, red};

    for (int c = 0; c < nchunk; ++c) {
        const int tc0 = t_begin + c * kC;
        const int valid = min(kC, t_end - tc0);
        // (1) Q, K tiles -> fp16; key norms
        alive = alive && mbar_wait(&bars[1], ph_qk, kWaitLimit);
        ph_qk ^= 1;
        if (__syncthreads_or(!alive)) break;
        key_tile_prepare(xk, nd, nk, part);
        {
            float ss, am;
            convert_tile(xq, nd, ss, am);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // (2) P_K
        if (threadIdx.x == 0) {
            issue_projection(g, tmem, xk_s, w_s, g.nproj, 0, nft, 0);
            mma_commit(&bars[3]);
        }
        alive = mbar_wait(&bars[3], ph_m, kWaitLimit);
        ph_m ^= 1;
        if (__syncthreads_or(!alive)) break;
        tc_fence_after();
        // (3) key features (may raise the key reference)
        float mass;
        float alpha = key_features(g, tmem, 0, nft, phk, valid, ep, &mass);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // (4) P_Q
        if (threadIdx.x == 0) {
            issue_projection(g, tmem, xq_s, w_s, g.nproj, 0, nft, 0);
            mma_commit(&bars[3]);
        }
        alive = mbar_wait(&bars[3], ph_m, kWaitLimit);
        ph_m ^= 1;
        if (__syncthreads_or(!alive)) break;
        tc_fence_after();
        // (5) state -> fp16 operand (Q/K tiles are free now), z -> smem
        {
            float zmax = sc[1] * alpha;
            const float vmax = sc[2];
            const float bound = zmax * vmax;
            const float sigma = bound > 0.f ? exp2f(floorf(log2f(kSigmaTarget / bound))) : 1.f;
            for (int t = 0; t < nft; ++t) {
                const int f = t * 128 + row;
                float v[32];
                tmem_ld32(tm_addr(tmem, q, col_s + t * s_stride + 32 * h), v);
                tmem_ld_wait();
                if (alpha != 1.f) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= alpha;
                    tmem_st32(tm_addr(tmem, q, col_s + t * s_stride + 32 * h), v);
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= sigma;
                store_row32(sop, f, 32 * h, v);
                if (h == 0) {
                    float zv[32];
                    tmem_ld32(tm_addr(tmem, q, col_s + t * s_stride + 64), zv);
                    tmem_ld_wait();
                    const float zval = zv[0] * alpha;
                    zs[f] = zval;
                    if (alpha != 1.f) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) zv[i] = zval;
                        tmem_st32(tm_addr(tmem, q, col_s + t * s_stride + 64), zv);
                    }
                }
            }
            tmem_st_wait();
            if (threadIdx.x == 0) {
                sc[1] = zmax + mass;   // bound on max_f z_f after this chunk's update
                sc[4] = sigma;
            }
        }
        fence_async_smem();
        __syncthreads();
        const float sigma = sc[4];
        // (6) query features (+ phi_q . z)
        float den = query_features(g, tmem, phq, zs, part);
        dpart[h * 128 + row] = den;
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // (7) A = phi_Q phi_K^T, D_inter = phi_Q S_op
        if (threadIdx.x == 0) {
            const uint32_t idesc = idesc_f16(128, 128, 0, 0);
            for (int kk = 0; kk < g.r / 16; ++kk) {
                uint64_t aa = smem_desc(phq_s + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
                uint64_t bb = smem_desc(phk_s + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
                mma_f16(tmem + col_a, aa, bb, idesc, kk > 0);
            }
            issue_inter(g, tmem + col_di, phq_s, sop_s, 0);
            mma_commit(&bars[3]);
        }
        alive = mbar_wait(&bars[3], ph_m, kWaitLimit);
        ph_m ^= 1;
        if (__syncthreads_or(!alive)) break;
        tc_fence_after();
        // Q/K tiles and the state operand are free: prefetch the next chunk's Q, K
        if (threadIdx.x == 0 && c + 1 < nchunk) {
            mbar_arrive_expect_tx(&bars[1], 2 * kBlk * nd);
            for (int b = 0; b < nd; ++b) {
                tma_load_3d(xq + b * kBlk, &tm_q, &bars[1], 64 * b, tc0 + kC, bh);
                tma_load_3d(xk + b * kBlk, &tm_k, &bars[1], 64 * b, tc0 + kC, bh);
            }
        }
        // (8) intra-chunk matrix: causal mask, row sums, per-row power-of-two scale
        {
            float s = 0.f, mx = 0.f;
            for (int cc = 0; cc < 2; ++cc) {
                float v[32];
                tmem_ld32(tm_addr(tmem, q, col_a + 64 * h + 32 * cc), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int j = 64 * h + 32 * cc + i;
                    float x = (j <= row && j < valid) ? v[i] : 0.f;
                    s += x;
                    mx = fmaxf(mx, fabsf(x));
                }
            }
            part[h * 128 + row] = s;
            __syncthreads();
            const float rs = part[row] + part[128 + row];
            __syncthreads();
            part[h * 128 + row] = mx;
            __syncthreads();
            const float rm = fmaxf(part[row], part[128 + row]);
            const float r_scale = rm > 0.f ? exp2f(-floorf(log2f(rm))) : 1.f;
            if (h == 0) {
                deni[row] = rs;
                rho[row] = r_scale;
            }
            uint8_t *blk = bhat + (size_t)h * kBlk;
            for (int cc = 0; cc < 2; ++cc) {
                float v[32];
                tmem_ld32(tm_addr(tmem, q, col_a + 64 * h + 32 * cc), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int j = 64 * h + 32 * cc + i;
                    v[i] = (j <= row && j < valid) ? v[i] * r_scale : 0.f;
                }
                store_row32(blk, row, 32 * cc, v);
            }
        }
        // V tile -> fp16, running max |v|
        alive = alive && mbar_wait(&bars[2], ph_v, kWaitLimit);
        ph_v ^= 1;
        if (__syncthreads_or(!alive)) break;
        {
            float ss, am;
            convert_tile(xv, 1, ss, am);
            const float vm = cta_max(am, red);
            if (threadIdx.x == 0) sc[2] = fmaxf(sc[2], vm);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // (9) D_intra = B V ; S += phi_K^T V ; z += phi_K^T 1
        if (threadIdx.x == 0) {
            const uint32_t idesc = idesc_f16(128, 64, 0, 1);
            for (int kk = 0; kk < kC / 16; ++kk) {
                uint64_t aa = smem_desc(bhat_s + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
                uint64_t bb = smem_desc(xv_s + kk * 2048, kBlk, 1024);
                mma_f16(tmem + col_da, aa, bb, idesc, kk > 0);
            }
            issue_state_update(tmem, phk_s, xv_s, ones_s, nft, col_s, s_stride, 1);
            mma_commit(&bars[3]);
        }
        alive = mbar_wait(&bars[3], ph_m, kWaitLimit);
        ph_m ^= 1;
        if (__syncthreads_or(!alive)) break;
        tc_fence_after();
        if (threadIdx.x == 0 && c + 1 < nchunk) {
            mbar_arrive_expect_tx(&bars[2], kBlk);
            tma_load_3d(xv, &tm_v, &bars[2], 64 * dvt, tc0 + kC, bh);
        }
        // (10) out = (D_intra / rho + D_inter / sigma) / (den_intra + den_inter)
        {
            float di[32], da[32];
            tmem_ld32(tm_addr(tmem, q, col_da + 32 * h), da);
            tmem_ld32(tm_addr(tmem, q, col_di + 32 * h), di);
            tmem_ld_wait();
            const float dn = deni[row] + dpart[row] + dpart[128 + row];
            const float inv = 1.f / dn, ia = 1.f / rho[row], is = 1.f / sigma;
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = fmaf(da[i], ia, di[i] * is) * inv;
            stage_out(stage, row, h, o);
        }
        fence_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            tma_store_3d(&tm_out, stage, 64 * dvt, tc0, bh);
            tma_store_3d(&tm_out, stage + kBlk, 64 * dvt + 32, tc0, bh);
            bulk_commit();
            bulk_wait_read0();   // phi_K of the next chunk reuses the staging area
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) bulk_wait0();
    if (!alive) set_status(a.status, FAVOR_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, a.tmem_cols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
constexpr uint32_t kSmemMax = 232448;   // 227 KB opt-in per block

uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }

Geo make_geo(const Problem &p) {
    Geo g;
    g.d = p.d;
    g.dv = p.dv;
    g.r = p.r;
    g.nproj = p.nproj;
    g.map = p.map;
    g.n_ft = p.r / 128;
    g.np_tile = p.map == FAVOR_MAP_TRIG ? 64 : 128;
    return g;
}

struct CausalLayout {
    uint32_t o_w, o_xq, o_xk, o_xv, o_phq, o_phk, o_ones, o_small, bytes;
};
CausalLayout causal_layout(const Geo &g) {
    CausalLayout l;
    uint32_t o = 0;
    l.o_w = o; o = align1k(o + (uint32_t)g.nproj * g.d * 2);
    l.o_xq = o; o = align1k(o + (uint32_t)kC * g.d * 2);
    l.o_xk = o; o = align1k(o + (uint32_t)kC * g.d * 2);
    l.o_xv = o; o = align1k(o + kBlk);
    l.o_phq = o; o = align1k(o + (uint32_t)kC * g.r * 2);
    l.o_phk = o; o = align1k(o + (uint32_t)kC * g.r * 2);
    l.o_ones = o; o = align1k(o + 4096);
    l.o_small = o; o = align1k(o + 1200 * 4);
    l.bytes = o + 1024;
    return l;
}

struct StateLayout {
    uint32_t o_w, o_xk, o_xv, o_phk, o_ones, o_small, bytes;
};
StateLayout state_layout(const Geo &g) {
    StateLayout l;
    uint32_t o = 0;
    l.o_w = o; o = align1k(o + (uint32_t)g.np_tile * g.d * 2);
    l.o_xk = o; o = align1k(o + (uint32_t)kC * g.d * 2);
    l.o_xv = o; o = align1k(o + (uint32_t)kC * g.dv * 2);
    l.o_phk = o; o = align1k(o + 2 * kBlk);
    l.o_ones = o; o = align1k(o + 4096);
    l.o_small = o; o = align1k(o + 420 * 4);
    l.bytes = o + 1024;
    return l;
}

struct OutputLayout {
    uint32_t o_w, o_xq, o_sop, o_phq, o_stage, o_small, bytes;
};
OutputLayout output_layout(const Geo &g) {
    OutputLayout l;
    uint32_t o = 0;
    l.o_w = o; o = align1k(o + (uint32_t)g.nproj * g.d * 2);
    l.o_xq = o; o = align1k(o + (uint32_t)kC * g.d * 2);
    l.o_sop = o; o = align1k(o + (uint32_t)g.r * 128);
    l.o_phq = o; o = align1k(o + (uint32_t)kC * g.r * 2);
    l.o_stage = o; o = align1k(o + 2 * kBlk);
    l.o_small = o; o = align1k(o + 800 * 4);
    l.bytes = o + 1024;
    return l;
}

int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 148;
        }
    }
    return n;
}

}  // namespace

bool tc_supported(const Problem &p) {
    if (p.d != 64 && p.d != 128) return false;
    if (p.dv != 64 && p.dv != 128) return false;
    if (p.r != 128 && p.r != 256) return false;
    if (p.map == FAVOR_MAP_ELU1 && p.r != 128) return false;
    Geo g = make_geo(p);
    if (p.causal) {
        if (causal_layout(g).bytes > kSmemMax) return false;
    } else {
        if (output_layout(g).bytes > kSmemMax) return false;
    }
    if (state_layout(g).bytes > kSmemMax) return false;
    return encoder() != nullptr;
}

namespace {
struct Plan {
    int G, seg_len, nstate, nvb, nchunk;
    size_t img_bytes, per_state, bytes;
};

Plan make_plan(const Problem &p) {
    const Geo g = make_geo(p);
    Plan pl;
    pl.nvb = p.dv / 64;
    pl.nchunk = (p.L + kC - 1) / kC;
    const int sms = num_sms();
    // segments: whole 128-token chunks, about one CTA per SM in the scan
    int G;
    if (p.causal) {
        G = (int)std::lround((double)sms / (p.BH * pl.nvb));
    } else {
        G = (int)std::lround(2.0 * sms / (p.BH * g.n_ft));
    }
    G = std::max(1, std::min(G, pl.nchunk));
    const int seg_chunks = (pl.nchunk + G - 1) / G;
    pl.G = (pl.nchunk + seg_chunks - 1) / seg_chunks;
    pl.seg_len = seg_chunks * kC;
    pl.nstate = p.causal ? pl.G - 1 : pl.G;
    pl.img_bytes = (size_t)p.H * p.nproj * p.d * 2;
    pl.per_state = (size_t)p.r * (p.dv + 1);
    size_t bytes = carve_bytes<uint8_t>(pl.img_bytes) +
                   carve_bytes<float>((size_t)p.BH * std::max(1, pl.nstate) * pl.per_state) +
                   carve_bytes<float>((size_t)p.BH * std::max(1, pl.nstate) * g.n_ft * 4);
    if (p.causal)
        bytes += carve_bytes<float>((size_t)p.BH * pl.G * pl.per_state) +
                 carve_bytes<float>((size_t)p.BH * pl.G * 4);
    else
        bytes += carve_bytes<uint8_t>((size_t)p.BH * pl.nvb * p.r * 128) +
                 carve_bytes<float>((size_t)p.BH * p.r) + carve_bytes<float>(p.BH);
    pl.bytes = bytes;
    return pl;
}
}  // namespace

size_t tc_scratch_bytes(const Problem &p) { return make_plan(p).bytes; }

int tc_forward(const void *q, const void *k, const void *v, const float *omega, float *out,
               const Problem &p, cudaStream_t st) {
    int status = FAVOR_OK;
    const size_t bytes = tc_scratch_bytes(p);
    void *ws = workspace(bytes, &status);
    if (!ws) return status;
    return tc_run(q, k, v, omega, out, p, st, ws, bytes);
}

int tc_run(const void *q, const void *k, const void *v, const float *omega, float *out,
           const Problem &p, cudaStream_t st, void *ws, size_t ws_bytes) {
    const Geo g = make_geo(p);
    const Plan pl = make_plan(p);
    if (ws_bytes < pl.bytes) return FAVOR_ERR_UNSUPPORTED;
    const int nvb = pl.nvb, nchunk = pl.nchunk, G = pl.G, seg_len = pl.seg_len,
              nstate = pl.nstate;
    const int sms = num_sms();
    const size_t img_bytes = pl.img_bytes, per_state = pl.per_state;
    int *dstat = device_status_ptr();
    Carve cv{static_cast<char *>(ws), 0};
    uint8_t *img = cv.take<uint8_t>(img_bytes);
    float *state = cv.take<float>((size_t)p.BH * std::max(1, nstate) * per_state);
    float *meta = cv.take<float>((size_t)p.BH * std::max(1, nstate) * g.n_ft * 4);

    CUtensorMap mq, mk, mv, mo;
    int rc;
    if ((rc = make_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.BH, p.L, p.d, 64)) ||
        (rc = make_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.BH, p.L, p.d, 64)) ||
        (rc = make_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.BH, p.L, p.dv, 64)) ||
        (rc = make_map(&mo, out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.BH, p.L, p.dv, 32)))
        return rc;

    tc_prep_omega<<<dim3(32, p.H), 256, 0, st>>>(omega, img, p.H, p.nproj, p.d, p.map);
    FAVOR_LAUNCH_CHECK();

    if (nstate > 0) {
        StateLayout sl = state_layout(g);
        StateArgs sa;
        sa.g = g; sa.H = p.H; sa.L = p.L; sa.seg_len = seg_len; sa.nseg = nstate;
        sa.omg = img; sa.state = state; sa.meta = meta; sa.status = dstat;
        sa.o_w = sl.o_w; sa.o_xk = sl.o_xk; sa.o_xv = sl.o_xv; sa.o_phk = sl.o_phk;
        sa.o_ones = sl.o_ones; sa.o_small = sl.o_small;
        sa.tmem_cols = (128 + p.dv + 16) <= 256 ? 256 : 512;
        if (cudaFuncSetAttribute(tc_state, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sl.bytes) != cudaSuccess)
            return FAVOR_ERR_CUDA;
        tc_state<<<dim3(g.n_ft, nstate, p.BH), kThreads, sl.bytes, st>>>(mk, mv, sa);
        FAVOR_LAUNCH_CHECK();
    }

    if (!p.causal) {
        uint8_t *sop = cv.take<uint8_t>((size_t)p.BH * nvb * p.r * 128);
        float *z = cv.take<float>((size_t)p.BH * p.r);
        float *sig = cv.take<float>(p.BH);
        CombineArgs ca{};
        ca.g = g; ca.nseg = nstate; ca.causal = 0; ca.state = state; ca.meta = meta;
        ca.sop = sop; ca.zout = z; ca.sig = sig;
        tc_combine<<<dim3(p.BH, 1), 256, 0, st>>>(ca);
        FAVOR_LAUNCH_CHECK();
        OutputLayout ol = output_layout(g);
        OutputArgs oa;
        oa.g = g; oa.H = p.H; oa.L = p.L;
        const int want_ctas = 2 * sms;
        int per = std::max(1, (int)((long long)nchunk * p.BH * nvb / want_ctas));
        oa.chunks_per_cta = per;
        oa.omg = img; oa.sop = sop; oa.z = z; oa.sig = sig; oa.status = dstat;
        oa.o_w = ol.o_w; oa.o_xq = ol.o_xq; oa.o_sop = ol.o_sop; oa.o_phq = ol.o_phq;
        oa.o_stage = ol.o_stage; oa.o_small = ol.o_small; oa.tmem_cols = 512;
        if (cudaFuncSetAttribute(tc_output, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ol.bytes) != cudaSuccess)
            return FAVOR_ERR_CUDA;
        dim3 grid((nchunk + per - 1) / per, nvb, p.BH);
        stats_begin(st, "tc_output");
        tc_output<<<grid, kThreads, ol.bytes, st>>>(mq, mo, oa);
        stats_end(st);
        FAVOR_LAUNCH_CHECK();
        return FAVOR_OK;
    }

    float *s_in = cv.take<float>((size_t)p.BH * G * per_state);
    float *meta_in = cv.take<float>((size_t)p.BH * G * 4);
    if (G > 1) {
        CombineArgs ca{};
        ca.g = g; ca.nseg = nstate; ca.causal = 1; ca.state = state; ca.meta = meta;
        ca.s_in = s_in; ca.meta_in = meta_in;
        tc_combine<<<dim3(p.BH, G - 1), 256, 0, st>>>(ca);
        FAVOR_LAUNCH_CHECK();
    }
    CausalLayout cl = causal_layout(g);
    CausalArgs a;
    a.g = g; a.H = p.H; a.L = p.L; a.seg_len = seg_len; a.nseg = G;
    a.omg = img; a.s_in = s_in; a.meta_in = meta_in; a.status = dstat;
    a.o_w = cl.o_w; a.o_xq = cl.o_xq; a.o_xk = cl.o_xk; a.o_xv = cl.o_xv; a.o_phq = cl.o_phq;
    a.o_phk = cl.o_phk; a.o_ones = cl.o_ones; a.o_small = cl.o_small; a.tmem_cols = 512;
    if (cudaFuncSetAttribute(tc_causal, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cl.bytes) != cudaSuccess)
        return FAVOR_ERR_CUDA;
    stats_begin(st, "tc_causal");
    tc_causal<<<dim3(G, nvb, p.BH), kThreads, cl.bytes, st>>>(mq, mk, mv, mo, a);
    stats_end(st);
    FAVOR_LAUNCH_CHECK();
    return FAVOR_OK;
}

}  // namespace favor
