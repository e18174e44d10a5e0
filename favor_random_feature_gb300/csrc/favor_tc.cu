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
// Those offsets keep every fp16 feature at most e^10.  There is no lower
// bound: a key whose features lie far below the head's reference (about e^-18
// or more below its largest key feature so far) flushes to zero in fp16.  The
// kernels check the denominators they form against that flush level (and every
// operand against fp16's largest value) and report FAVOR_ERR_RANGE through the
// device status word when an input leaves the range.  The intra-chunk matrix
// is normalised per row by a power of two before it is rounded to fp16, and
// the state operand by a power of two bounded from the running key mass; both
// factors are divided out in fp32.
//
// Kernels: tc_prep_omega (fp16 image of W), tc_state (segment states),
// tc_combine (fixed-order sums / exclusive prefixes of the segment states),
// tc_output (non-causal rows), tc_causal (the chunked causal scan) and
// tc_causal_split (the same scan with a head's features split over the CTAs
// of a cluster).
#include <climits>
#include <cmath>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "favor_internal.h"
#include "tc_ptx.cuh"

namespace favor {
namespace {

using namespace tc;

constexpr int kC = 128;                 // tokens per chunk (= MMA M)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kShift = 8.0f * 1.4426950408889634f;   // e^8 headroom (log2 units)
constexpr float kSigmaTarget = 16384.f;  // bound for |sigma * S| in the fp16 state operand
// largest key feature kept, e^10: a chunk may exceed the reference by e^2
// before the reference moves
constexpr float kLog2MaxFeature = 14.4269504f;          // log2(e^10)
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

// 3D map over a [BH][L][cols] tensor, box [1][box_rows][box_cols], 128B swizzle.
int make_map(CUtensorMap *m, const void *base, CUtensorMapDataType type, int esize, int BH, int L,
             int cols, int box_cols, int box_rows = kC) {
    auto enc = encoder();
    if (!enc) return FAVOR_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)L, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)cols * esize, (cuuint64_t)L * cols * esize};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
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

// 2^-floor(log2 x) for a positive normal x: the exponent field, negated
__device__ __forceinline__ float pow2_inv_floor(float x) {
    return __int_as_float(0x7F000000 - (__float_as_int(x) & 0x7F800000));
}

// the largest power of two s with s * b <= 2^14 (b > 0 normal): 2^(14 - ceil(log2 b))
__device__ __forceinline__ float pow2_scale_14(float b) {
    const int bits = __float_as_int(b);
    const int e = ((bits >> 23) & 0xFF) - 127 + ((bits & 0x7FFFFF) ? 1 : 0);
    const int se = min(max(14 - e, -126), 127);
    return __int_as_float((se + 127) << 23);
}

__device__ __forceinline__ void set_status(int *status, int code) {
    if (status) atomicExch(status, code);
}

// FAVOR_ERR_RANGE unless another error is already recorded: an input left
// the range of the fp16 operands (the call still completes)
__device__ __forceinline__ void flag_range(int *status) {
    if (status) atomicCAS(status, FAVOR_OK, FAVOR_ERR_RANGE);
}

// the largest |x| that bf16 -> fp16 conversion keeps finite: 65280, the
// largest bf16 value below fp16's 65504 (inf and larger values fail the test)
constexpr float kMaxOperand = 65280.f;
// The fp16 floor of a positive-feature denominator: every operand feature
// carries an absolute rounding error of at most 2^-25 (subnormal spacing
// 2^-24, halved), so a row whose denominator is below (keys) x (row sum of
// its query features) x 2^-15 may have lost more than 2^-10 of it to
// underflow.  For inputs inside the range this ratio stays above 2^-9.
constexpr float kRangeFloor = 3.0517578125e-05f;   // 2^-15

// A bounded wait made to run out: one thread waits for the first phase of an
// mbarrier that nothing arrives on, with the same bounded wait the pipelines
// use.  It gives up after `limit` clock cycles and records the expiry the way
// a stalled pipeline does, so the expiry path and the status word can be
// checked without faulting or hanging anything.
__global__ void __launch_bounds__(1) wait_expiry_kernel(int *status, long long limit) {
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, limit)) set_status(status, FAVOR_ERR_TIMEOUT);
}

// sin/cos with the argument first reduced to [-pi, pi] (Cody-Waite) so that
// the hardware approximations stay accurate for projections of any size met
// here.  2pi = p1 + p2 + p3: p1 = 6.28125 has 8 significant bits, so n p1 is
// exact for |n| < 2^16; p2 = fl(2pi - p1) and p3 = fl(2pi - p1 - p2), which
// leaves a representation error of about 3e-19 per period.
__device__ __forceinline__ void sincos_reduced(float x, float &s, float &c) {
    const float inv2pi = 0.15915494309189535f;
    const float p1 = 6.28125f, p2 = 1.935307169e-3f, p3 = 1.025337627e-11f;
    float n = rintf(x * inv2pi);
    float t = fmaf(-n, p1, x);
    t = fmaf(-n, p2, t);
    t = fmaf(-n, p3, t);
    __sincosf(t, &s, &c);
}

// ELU + 1 ("Kernel Feature Maps" section 1); p is x itself here.
__device__ __forceinline__ float elu1(float p) { return p > 0.f ? p + 1.f : ex2(p * kLog2e); }

// sincos_reduced on n arguments, for the accuracy test of the reduction
__global__ void sincos_check_kernel(const float *__restrict__ x, float *__restrict__ s, float *__restrict__ c,
                                    int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        sincos_reduced(x[i], s[i], c[i]);
}

// ---------------------------------------------------------------------------
// W image: fp16, 128B-swizzled MN-major atoms [d][64] per 64 projections
// (the B operand of P = X W^T with K = d), scaled by log2(e) for the
// positive map; the identity for elu1.
// ---------------------------------------------------------------------------
// rows: rows of the caller's omega per head; projection p takes row p % rows
// (rows < nproj: a widened head, every projection twice)
__global__ void tc_prep_omega(const float *__restrict__ omega, uint8_t *__restrict__ img, int H,
                              int nproj, int d, int map, int rows) {
    grid_dep_launch();
    const int h = blockIdx.y;
    const size_t per = (size_t)nproj * d;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < per;
         e += (size_t)gridDim.x * blockDim.x) {
        int p = (int)(e / d), j = (int)(e % d);
        const int src = p % rows;
        float w;
        if (map == FAVOR_MAP_ELU1) w = (src == j) ? 1.f : 0.f;
        else w = omega[((size_t)h * rows + src) * d + j] * (map == FAVOR_MAP_POSITIVE ? kLog2e : 1.f);
        uint8_t *atom = img + (size_t)h * per * 2 + (size_t)(p / 64) * d * 128;
        *reinterpret_cast<__half *>(atom + sw128_offset(j, p % 64)) = __float2half_rn(w);
    }
}

// ---------------------------------------------------------------------------
// Epilogue group helpers (tc_state, tc_causal, tc_output): warps 1..16 of a
// CTA, 512 threads synchronised on named barrier 1.
// ---------------------------------------------------------------------------
constexpr int kEpi = 512;

__device__ __forceinline__ float grp_max(float v, float *red, int ew) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    group_sync(kEpi);
    if ((threadIdx.x & 31) == 0) red[ew] = v;
    group_sync(kEpi);
    float r = red[0];
#pragma unroll
    for (int i = 1; i < kEpi / 32; ++i) r = fmaxf(r, red[i]);
    return r;
}

// Bounded mbarrier wait that also gives up at once when another thread of
// the CTA has already timed out (*abort set), so that every thread keeps
// running the same sequence of group barriers and the kernel still ends.
__device__ __forceinline__ bool ewait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    // later polls suspend in hardware until the phase completes (at most
    // 100 us each), so a waiting warp leaves the issue slots to the others
    while (!mbar_try_wait_hint(bar, parity, 100000u)) {
        if (*abort) return false;
        if (clock64() - t0 > kWaitLimit) {
            *abort = 1;
            return false;
        }
    }
    return true;
}

// ewait for an mbarrier that other CTAs of the cluster complete (remote
// stores, remote arrivals): the wait acquires at cluster scope.
__device__ __forceinline__ bool cwait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    const long long t0 = clock64();
    while (!mbar_try_wait_cluster(bar, parity)) {
        if (*abort) return false;
        if (clock64() - t0 > kWaitLimit) {
            *abort = 1;
            return false;
        }
    }
    return true;
}

// In-place bf16 -> fp16 conversion of a [128][64 nblk] tile by 512 threads:
// thread e converts two 16-byte chunks of row e % 128 per block (chunk index
// rotated with the row).  SQ / AMAX select the statistics it also returns:
// the partial sum of squares (key norms) and max |x| (values).
template <bool SQ, bool AMAX>
__device__ __forceinline__ float convert_tile_512(uint8_t *tile, int nblk, int e, float &amax) {
    const int row = e & 127, part = e >> 7;
    float sumsq = 0.f;
    amax = 0.f;
    for (int b = 0; b < nblk; ++b) {
        uint8_t *rp = tile + b * kBlk + row * 128;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int p = (part * 2 + c + row) & 7;
            uint4 *ptr = reinterpret_cast<uint4 *>(rp + p * 16);
            uint4 u = *ptr;
            uint32_t w[4] = {u.x, u.y, u.z, u.w}, o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
                if (SQ) sumsq = fmaf(lo, lo, fmaf(hi, hi, sumsq));
                if (AMAX) amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
                o[i] = pack_half2(lo, hi);
            }
            *ptr = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    return sumsq;
}

// One 16-byte chunk (8 values) of a bf16 tile -> fp16 in place; returns the
// chunk's sum of squares and raises amax to the chunk's largest |x|.
__device__ __forceinline__ float cvt_chunk16_sq(uint8_t *p, float &amax) {
    uint4 u = *reinterpret_cast<uint4 *>(p);
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
        ss = fmaf(lo, lo, fmaf(hi, hi, ss));
        amax = fmax3(amax, fabsf(lo), fabsf(hi));
        w[i] = pack_half2(lo, hi);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    return ss;
}

// ---------------------------------------------------------------------------
// tc_state: per (feature group, piece, head) the state of a run of keys
//   S[f][c] = sum_t phi(k_t)_f v_t[c],  z[f] = sum_t phi(k_t)_f
// at the key reference R, written as fp32 [f][dv + 1] plus (R, max z,
// max|v|, max|S|) per 128-feature tile.  A CTA covers FT = 1 or 2 feature
// tiles (all of a head's features where TMEM holds them), so each K and V
// tile is converted once for all of them.
// Warp 0 lane 0 issues every TMA copy and MMA; warps 1..16 (the epilogue
// group) compute features, warp w on TMEM lane quarter w % 4 and projection
// quarter (w - 1) / 4; warps 17..20 (the converters, one thread per row)
// turn each K and V tile into fp16 in place as soon as it lands, with the key
// norms and the range checks.  The epilogue reads the projections of chunk c
// into registers and hands TMEM back at once, so the tensor core projects
// chunk c + 1 while the features of c are formed, and the state update of c
// runs while the epilogue starts on c + 1.
// ---------------------------------------------------------------------------
constexpr int kStateConv = 128;
constexpr int kStateThreads = 32 + kEpi + kStateConv;

struct StateArgs {
    Geo g;
    int H, L, FT, piece_len, npieces, nvs, nks; // piece p: tokens [p piece_len, (p+1) piece_len) within L
    const uint8_t *omg;                // MN-major W images
    float *state;                      // [BH][npieces][r][dv+1]
    float *meta;                       // [BH][npieces][n_ft][4]: R, max z, max|v|, max|S|
    int *status;
    uint32_t o_w, o_xk, o_xv, o_phk, o_small, xv_stride, tmem_cols;
};

// N fp16 values (packed pairs) of one row into 128B-swizzled [128][64]
// blocks at columns [c0, c0 + N)
template <int N>
__device__ __forceinline__ void store_row_packed(uint8_t *blk, int row, int c0, const uint32_t *h) {
#pragma unroll
    for (int c = 0; c < N / 8; ++c)
        *reinterpret_cast<uint4 *>(blk + sw128_offset(row, c0 + 8 * c)) =
            make_uint4(h[4 * c + 0], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
}

// NC consecutive TMEM columns of the thread's lane into registers
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&pv)[NC]) {
    if constexpr (NC % 32 == 0) {
#pragma unroll
        for (int b = 0; b < NC / 32; ++b) {
            float t[32];
            tmem_ld32(taddr + 32 * b, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) pv[32 * b + i] = t[i];
        }
    } else {
        static_assert(NC == 16, "16, 32 or 64 columns");
        float t[16];
        tmem_ld16(taddr, t);
#pragma unroll
        for (int i = 0; i < 16; ++i) pv[i] = t[i];
    }
}

// NC = projection columns per epilogue thread (a quarter of the group's
// projections), MAP the feature map
template <int NC, int MAP>
__device__ __forceinline__ void state_body(const CUtensorMap *tm_k, const CUtensorMap *tm_v, const StateArgs &a,
                                           uint8_t *sm) {
    const Geo &g = a.g;
    const int FT = a.FT, fg = blockIdx.x, piece = blockIdx.y, bh = blockIdx.z, head = bh % a.H;
    const int t_begin = piece * a.piece_len, t_end = min(a.L, t_begin + a.piece_len);
    const int nchunk = max(0, (t_end - t_begin + kC - 1) / kC);
    const int nd = g.d / 64, nvb = g.dv / 64, NSV = a.nvs, NSK = a.nks;
    const int npg = FT * g.np_tile;                  // projections of the group
    const uint32_t xkb = (uint32_t)kC * g.d * 2;
    uint8_t *w = sm + a.o_w, *xk = sm + a.o_xk, *xv = sm + a.o_xv, *phk = sm + a.o_phk;
    float *small = reinterpret_cast<float *>(sm + a.o_small);
    float *nk = small;              // [3][128] half key norms, by chunk % 3
    float *cred = small + 384;      // [4] the converters' max |v|
    float *red = small + 768;       // [32]
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + 800);
    // e_x: K(c) converted, one barrier per K buffer (c % NSK): the converters
    // may run NSK tiles ahead of the thread that waits, and a barrier must not
    // complete twice before it looks.  e_n: the norms of chunk c (by c % 3,
    // the slot they use).  e_v: V(c) converted (by c % 2; NSV <= 2).
    uint64_t *bar_w = &bars[0], *bar_pk = &bars[1], *bar_s = &bars[2], *bar_v = &bars[3] /*[2]*/,
             *bar_k = &bars[5] /*[3]*/, *e_x = &bars[8] /*[3]*/, *e_pk = &bars[11], *e_k = &bars[12],
             *e_n = &bars[13] /*[3]*/, *e_v = &bars[16] /*[2]*/;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(small + 836);
    volatile int *abortp = reinterpret_cast<volatile int *>(small + 838);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col_s = 256;          // state tile t at col_s + t (dv + 16): dv values, then 16 copies of z
    const int sw = g.dv + 16;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 8; ++i) mbar_init(&bars[i], 1);
        for (int i = 8; i < 11; ++i) mbar_init(&bars[i], kStateConv);
        for (int i = 11; i < 13; ++i) mbar_init(&bars[i], kEpi);
        for (int i = 13; i < 18; ++i) mbar_init(&bars[i], kStateConv);
        fence_mbar_init();
        *abortp = 0;
    }
    // ones atom after the V blocks of each V buffer (the z column)
    for (int s = 0; s < NSV; ++s) {
        uint8_t *ones = xv + (size_t)s * a.xv_stride + (size_t)nvb * kBlk;
        for (int i = threadIdx.x; i < (int)(kBlk / 16); i += kStateThreads)
            reinterpret_cast<uint4 *>(ones)[i] = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    }
    if (warp == 0) tmem_alloc(tslot, a.tmem_cols);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool alive = true;
    grid_dep_launch();

    if (warp == 0) {
        if (lane == 0 && nchunk == 0) grid_dep_wait();
        if (lane == 0 && nchunk > 0) {
            const uint32_t w_s = smem_u32(w), xk_s = smem_u32(xk), xv_s = smem_u32(xv), phk_s = smem_u32(phk);
            const uint32_t wbytes = (uint32_t)npg * g.d * 2;
            auto load_k = [&](int c) {
                uint64_t *bar = &bar_k[c % NSK];
                mbar_arrive_expect_tx(bar, xkb);
                for (int b = 0; b < nd; ++b)
                    tma_load_3d(xk + (size_t)(c % NSK) * xkb + b * kBlk, tm_k, bar, 64 * b, t_begin + c * kC, bh);
            };
            auto load_v = [&](int c) {
                const int s = c % NSV;
                mbar_arrive_expect_tx(&bar_v[s], (uint32_t)nvb * kBlk);
                for (int b = 0; b < nvb; ++b)
                    tma_load_3d(xv + (size_t)s * a.xv_stride + b * kBlk, tm_v, &bar_v[s], 64 * b, t_begin + c * kC, bh);
            };
            auto issue_proj = [&](int c) {
                const uint32_t idesc = idesc_f16(128, npg, 0, 1);
                const uint32_t x_s = xk_s + (uint32_t)(c % NSK) * xkb;
                for (int kk = 0; kk < g.d / 16; ++kk)
                    mma_f16(tmem, smem_desc(x_s + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024),
                            smem_desc(w_s + kk * 2048, (uint32_t)g.d * 128, 1024), idesc, kk > 0);
                mma_commit(bar_pk);
            };
            for (int c = 0; c < min(NSK, nchunk); ++c) load_k(c);
            for (int c = 0; c < min(NSV, nchunk); ++c) load_v(c);
            // the W image comes from the kernel before this one
            grid_dep_wait();
            mbar_arrive_expect_tx(bar_w, wbytes);
            bulk_load(w, a.omg + (size_t)head * g.nproj * g.d * 2 + (size_t)fg * wbytes, wbytes, bar_w);
            alive = ewait(bar_w, 0, abortp) && ewait(&e_x[0], 0, abortp);
            if (alive) {
                tc_fence_after();
                issue_proj(0);
            }
            for (int c = 0; c < nchunk && alive; ++c) {
                if (c + 1 < nchunk) {
                    // the epilogue holds P(c) in registers (so P(c) is done and
                    // K buffer c % NSK is free) and has converted K(c + 1)
                    if (!(alive = ewait(e_pk, c & 1, abortp) &&
                                  ewait(&e_x[(c + 1) % NSK], ((c + 1) / NSK) & 1, abortp)))
                        break;
                    tc_fence_after();
                    issue_proj(c + 1);
                    if (c + NSK < nchunk) load_k(c + NSK);
                }
                if (!(alive = ewait(e_k, c & 1, abortp) && ewait(&e_v[c & 1], (c >> 1) & 1, abortp))) break;
                tc_fence_after();
                {
                    const uint32_t idesc = idesc_f16(128, sw, 1, 1);
                    const uint32_t b_s = xv_s + (uint32_t)(c % NSV) * a.xv_stride;
                    for (int t = 0; t < FT; ++t) {
                        const uint32_t a_s = phk_s + (uint32_t)t * 2 * kBlk;
                        for (int kk = 0; kk < kC / 16; ++kk)
                            mma_f16(tmem + col_s + t * sw, smem_desc(a_s + kk * 2048, kBlk, 1024),
                                    smem_desc(b_s + kk * 2048, kBlk, 1024), idesc, 1);
                    }
                    mma_commit(bar_s);
                }
                if (c + NSV < nchunk) {
                    if (!(alive = ewait(bar_s, c & 1, abortp))) break;
                    load_v(c + NSV);
                }
            }
            if (!alive) set_status(a.status, FAVOR_ERR_TIMEOUT);
        }
    } else if (warp > kEpi / 32) {
        // converters: thread r owns row r of every K and V tile; K(c + 1)
        // comes before V(c) (the projection of c + 1 is wanted first)
        const int r = threadIdx.x - 32 - kEpi;
        float vmax = 0.f;
        auto convert_k = [&](int c) {
            alive &= ewait(&bar_k[c % NSK], (c / NSK) & 1, abortp);
            uint8_t *tile = xk + (size_t)(c % NSK) * xkb + r * 128;
            float ss = 0.f, kmax = 0.f;
            for (int b = 0; b < nd; ++b)
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) ss += cvt_chunk16_sq(tile + b * kBlk + ((ch ^ (r & 7)) << 4), kmax);
            if (kmax > kMaxOperand) flag_range(a.status);
            nk[(c % 3) * 128 + r] = 0.5f * kLog2e * ss;
            fence_async_smem();
            mbar_arrive(&e_x[c % NSK]);
            mbar_arrive(&e_n[c % 3]);
        };
        auto convert_v = [&](int c) {
            alive &= ewait(&bar_v[c % NSV], (c / NSV) & 1, abortp);
            uint8_t *tile = xv + (size_t)(c % NSV) * a.xv_stride + r * 128;
            for (int b = 0; b < nvb; ++b)
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint4 *p4 = reinterpret_cast<uint4 *>(tile + b * kBlk + ((ch ^ (r & 7)) << 4));
                    const uint4 u = *p4;
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
                    uint32_t o[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float lo = __uint_as_float(w4[i] << 16), hi = __uint_as_float(w4[i] & 0xffff0000u);
                        vmax = fmax3(vmax, fabsf(lo), fabsf(hi));
                        o[i] = pack_half2(lo, hi);
                    }
                    *p4 = make_uint4(o[0], o[1], o[2], o[3]);
                }
            fence_async_smem();
            mbar_arrive(&e_v[c & 1]);
        };
        if (nchunk > 0) convert_k(0);
        for (int c = 0; c < nchunk; ++c) {
            if (c + 1 < nchunk) convert_k(c + 1);
            convert_v(c);
        }
        // max |v| of the piece for the epilogue's meta and the range check
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
        if (lane == 0) cred[r >> 5] = vmax;
        named_sync(2, kEpi + kStateConv);
        if (!alive) set_status(a.status, FAVOR_ERR_TIMEOUT);
    } else {
        const int e = threadIdx.x - 32, ew = e >> 5;
        const int q = (ew + 1) & 3, j = ew >> 2;
        const int row = q * 32 + lane;
        float R = MAP == FAVOR_MAP_POSITIVE ? -INFINITY : 0.f;
        // zero state and z
        {
            uint32_t zero[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) zero[i] = 0u;
            for (int t = 0; t < FT; ++t)
                for (int cc = 16 * j; cc < sw; cc += 64) tmem_st16(tm_addr(tmem, q, col_s + t * sw + cc), zero);
            tmem_st_wait();
        }
        for (int c = 0; c < nchunk; ++c) {
            const int tc0 = t_begin + c * kC;
            const int valid = min(kC, t_end - tc0);
            const bool ok = row < valid;
            // P(c) -> registers (for the positive map after a first pass that
            // only takes the row maximum, so that the vote below holds no
            // projections); TMEM then goes back to the tensor core for P(c + 1)
            float pv[NC];
            alive &= ewait(bar_pk, c & 1, abortp);
            tc_fence_after();
            auto take_p = [&]() {
                tmem_ld_cols<NC>(tm_addr(tmem, q, NC * j), pv);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(e_pk);
            };
            float mx = -INFINITY;
            if (MAP == FAVOR_MAP_POSITIVE) {
                tmem_ld_cols<NC>(tm_addr(tmem, q, NC * j), pv);
                tmem_ld_wait();
                mx = max_of<NC>(pv);
            } else {
                take_p();
            }
            // features of chunk c, packed fp16 pairs
            constexpr int NH = MAP == FAVOR_MAP_TRIG ? NC : NC / 2;
            uint32_t hp[NH];
            float alpha = 1.f;
            if (MAP == FAVOR_MAP_POSITIVE) {
                alive &= ewait(&e_n[c % 3], (c / 3) & 1, abortp);
                const float nkr = nk[(c % 3) * 128 + row];
                // a key whose largest feature would pass e^(shift + slack) at the
                // current reference (always so before the first key) moves the
                // reference to it; the running state is rescaled to match
                if (group_or(ok && mx - nkr - R > kLog2MaxFeature, kEpi)) {
                    const float Rn = grp_max(ok ? mx - nkr : -INFINITY, red, ew) - kShift;
                    if (R != -INFINITY) alpha = ex2(R - Rn);
                    R = Rn;
                }
                // rows past the end take an infinite offset: their features are 0
                const float off = ok ? nkr + R : INFINITY;
                take_p();
#pragma unroll
                for (int i = 0; i < NC / 2; ++i) hp[i] = pack_half2(ex2(pv[2 * i] - off), ex2(pv[2 * i + 1] - off));
            } else if (MAP == FAVOR_MAP_TRIG) {
                // NC projections: sines in hp[0, NC/2), cosines in hp[NC/2, NC)
#pragma unroll
                for (int i = 0; i < NC / 2; ++i) {
                    float s0, c0, s1, c1;
                    sincos_reduced(pv[2 * i], s0, c0);
                    sincos_reduced(pv[2 * i + 1], s1, c1);
                    if (!ok) s0 = c0 = s1 = c1 = 0.f;
                    hp[i] = pack_half2(s0, s1);
                    hp[NC / 2 + i] = pack_half2(c0, c1);
                }
            } else {
#pragma unroll
                for (int i = 0; i < NC / 2; ++i)
                    hp[i] = ok ? pack_half2(elu1(pv[2 * i]), elu1(pv[2 * i + 1])) : 0u;
            }
            // phi_K and the state are free once the update of chunk c - 1 is done
            if (c >= 1) alive &= ewait(bar_s, (c - 1) & 1, abortp);
            tc_fence_after();
            // the running state moves to the new reference
            if (MAP == FAVOR_MAP_POSITIVE && alpha != 1.f) {
                for (int t = 0; t < FT; ++t)
                    for (int cc = 16 * j; cc < sw; cc += 64) {
                        float v[16];
                        tmem_ld16(tm_addr(tmem, q, col_s + t * sw + cc), v);
                        tmem_ld_wait();
                        uint32_t u[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(v[i] * alpha);
                        tmem_st16(tm_addr(tmem, q, col_s + t * sw + cc), u);
                    }
                tmem_st_wait();
            }
            if (MAP == FAVOR_MAP_TRIG) {
                // projection p of the group: tile p / 64, sine in block 2 (p / 64),
                // cosine in block 2 (p / 64) + 1, column p % 64
                const int p0 = NC * j;
                uint8_t *blk = phk + (size_t)(2 * (p0 / 64)) * kBlk;
                store_row_packed<NC>(blk, row, p0 % 64, hp);
                store_row_packed<NC>(blk + kBlk, row, p0 % 64, hp + NC / 2);
            } else {
                // feature f of the group in block f / 64, column f % 64
#pragma unroll
                for (int g32 = 0; g32 < NC / 32; ++g32) {
                    const int f0 = NC * j + 32 * g32;
                    store_row_packed<32>(phk + (size_t)(f0 / 64) * kBlk, row, f0 % 64, hp + 16 * g32);
                }
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(e_k);
        }
        // the last state update, then S, z -> global with each tile's max |S|
        // and max z.  The group's tiles are staged in shared memory (the K, V
        // and feature buffers are free now) as their global rows [FT][128][dv + 1]
        // (a warp's 32 rows fall on 32 different banks), then leave in one bulk copy.
        if (nchunk > 0) alive &= ewait(bar_s, (nchunk - 1) & 1, abortp);
        tc_fence_after();
        const bool write = alive && !*abortp;
        named_sync(2, kEpi + kStateConv);   // the converters' max |v|
        const float vm = fmaxf(fmaxf(cred[0], cred[1]), fmaxf(cred[2], cred[3]));
        if (e == 0 && vm > kMaxOperand) flag_range(a.status);
        float *stg = reinterpret_cast<float *>(xk);
        float smax[2] = {0.f, 0.f}, zval[2] = {0.f, 0.f};
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (t >= FT) break;
            float *srow = stg + ((size_t)t * 128 + row) * (g.dv + 1);
            for (int cc = 16 * j; cc < g.dv; cc += 64) {
                float v[16];
                tmem_ld16(tm_addr(tmem, q, col_s + t * sw + cc), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    smax[t] = fmaxf(smax[t], fabsf(v[i]));
                    srow[cc + i] = v[i];
                }
            }
            if (j == 0) {
                float v[16];
                tmem_ld16(tm_addr(tmem, q, col_s + t * sw + g.dv), v);
                tmem_ld_wait();
                zval[t] = fabsf(v[0]);
                srow[g.dv] = v[0];
            }
        }
        fence_async_smem();
        group_sync(kEpi);
        if (write && e == 0) {
            float *dst = a.state + (((size_t)bh * a.npieces + piece) * g.r + (size_t)fg * FT * 128) * (g.dv + 1);
            bulk_store(dst, stg, (uint32_t)FT * 128 * (g.dv + 1) * 4);
            bulk_commit();
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (t >= FT) break;
            const int ft = fg * FT + t;
            const float sm_all = grp_max(smax[t], red, ew);
            const float zm = grp_max(zval[t], red, ew);
            if (write && e == 0) {
                float *m = a.meta + (((size_t)bh * a.npieces + piece) * g.n_ft + ft) * 4;
                m[0] = R;
                m[1] = zm;
                m[2] = vm;
                m[3] = sm_all;
            }
        }
        if (write && e == 0) bulk_wait0();
        if (!write) set_status(a.status, FAVOR_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, a.tmem_cols);
}

__global__ void __launch_bounds__(kStateThreads, 1)
tc_state(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
         const StateArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int nc = a.FT * a.g.np_tile / 4;
    if (a.g.map == FAVOR_MAP_POSITIVE) {
        if (nc == 64) state_body<64, FAVOR_MAP_POSITIVE>(&tm_k, &tm_v, a, sm);
        else state_body<32, FAVOR_MAP_POSITIVE>(&tm_k, &tm_v, a, sm);
    } else if (a.g.map == FAVOR_MAP_TRIG) {
        if (nc == 32) state_body<32, FAVOR_MAP_TRIG>(&tm_k, &tm_v, a, sm);
        else state_body<16, FAVOR_MAP_TRIG>(&tm_k, &tm_v, a, sm);
    } else {
        state_body<32, FAVOR_MAP_ELU1>(&tm_k, &tm_v, a, sm);
    }
}

// ---------------------------------------------------------------------------
// tc_combine: fixed-order combination of piece states, rescaled to one key
// reference R* (the largest of the pieces'), grid (heads, outputs, slices):
//  non-causal: KV = sum_g S_g 2^(R_g - R*), z likewise; sigma is a power of
//    two with sigma * (bound on max |KV| and max z) <= 16384; writes the fp16
//    operand image of [sigma KV | sigma z]: nvb atoms [r][64] of KV and one
//    z atom (128B-swizzled MN-major).
//  causal (output s for segment s + 1): S_in = sum_{g <= s} ..., fp32
//    [r][dv+1], with (R*, bound on max z, max |v|).
// The bounds come from each segment tile's max z and max |S|.
// ---------------------------------------------------------------------------
struct CombineArgs {
    Geo g;
    int nseg;              // piece states available
    int pps;               // causal: pieces per scan segment
    int causal;
    int slice;             // per block: state elements (causal) or (feature, 8-column) units (non-causal)
    const float *state, *meta;
    uint8_t *sop;          // non-causal: [BH][nvb + 1][r][64] fp16 image
    float *s_in;           // causal: [BH][nout][r][dv+1]
    float *meta_in;        // causal: [BH][nout][4]
    int nout;              // causal: scan segments
};

constexpr int kCombineMaxTiles = 512;   // pieces x feature tiles: at most 64 x 8

__global__ void tc_combine(const CombineArgs a) {
    grid_dep_launch();
    grid_dep_wait();
    const Geo &g = a.g;
    const int bh = blockIdx.x;
    const int upto = a.causal ? (blockIdx.y + 1) * a.pps : a.nseg;   // pieces [0, upto)
    __shared__ float scale[kCombineMaxTiles];
    __shared__ float sh[4];   // R*, z bound, |S| bound, vmax
    __shared__ float msh[kCombineMaxTiles * 4];
    const int nsc = upto * g.n_ft;   // <= kCombineMaxTiles (checked on the host)
    {
        // the segment tiles' (R, max z, max|v|, max|S|), loaded by all threads at once
        const float *mg = a.meta + (size_t)bh * a.nseg * g.n_ft * 4;
        for (int i = threadIdx.x; i < nsc * 4; i += blockDim.x) msh[i] = mg[i];
        __syncthreads();
    }
    const float *meta = msh;
    if (threadIdx.x == 0) {
        float R = -INFINITY, vmax = 0.f;
        for (int i = 0; i < nsc; ++i) {
            R = fmaxf(R, meta[i * 4]);
            vmax = fmaxf(vmax, meta[i * 4 + 2]);
        }
        float zb = 0.f, sb = 0.f;
        for (int gi = 0; gi < upto; ++gi) {
            float zt = 0.f, st = 0.f;
            for (int t = 0; t < g.n_ft; ++t) {
                const float *m = meta + (gi * g.n_ft + t) * 4;
                float sc = 1.f;
                if (g.map == FAVOR_MAP_POSITIVE) sc = (m[0] == -INFINITY || R == -INFINITY) ? 0.f : ex2(m[0] - R);
                scale[gi * g.n_ft + t] = sc;
                zt = fmaxf(zt, m[1] * sc);
                st = fmaxf(st, m[3] * sc);
            }
            zb += zt;
            sb += st;
        }
        sh[0] = g.map == FAVOR_MAP_POSITIVE ? R : 0.f;
        sh[1] = zb;
        sh[2] = sb;
        sh[3] = vmax;
    }
    __syncthreads();
    const int W = g.dv + 1;
    const size_t per = (size_t)g.r * W;
    const float *st = a.state + (size_t)bh * a.nseg * per;
    const size_t e0 = (size_t)blockIdx.z * a.slice, e1 = min(per, e0 + a.slice);
    if (a.causal) {
        float *dst = a.s_in + ((size_t)bh * a.nout + blockIdx.y + 1) * per;
        for (size_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
            const int ftile = (int)(e / W) / 128;
            float sum = 0.f;
            for (int gi = 0; gi < upto; ++gi) sum += st[gi * per + e] * scale[gi * g.n_ft + ftile];
            dst[e] = sum;
        }
        if (blockIdx.z == 0 && threadIdx.x == 0) {
            float *m = a.meta_in + ((size_t)bh * a.nout + blockIdx.y + 1) * 4;
            m[0] = sh[0];
            m[1] = sh[1];
            m[2] = sh[3];
            m[3] = 0.f;
        }
        return;
    }
    const float sb = fmaxf(sh[2], sh[1]);
    const float sigma = sb > 0.f ? exp2f(floorf(log2f(kSigmaTarget / sb))) : 1.f;
    const int nvb = g.dv / 64;
    uint8_t *img = a.sop + (size_t)bh * (nvb + 1) * g.r * 128;
    // unit u = (feature f, group cg of 8 value columns; cg = dv / 8 is the z
    // column): the pieces' sum, scaled, rounded and stored as one 16-byte chunk
    const int ng = g.dv / 8 + 1;
    const size_t u0 = (size_t)blockIdx.z * a.slice, u1 = min((size_t)g.r * ng, u0 + a.slice);
    for (size_t u = u0 + threadIdx.x; u < u1; u += blockDim.x) {
        const int f = (int)(u / ng), cg = (int)(u % ng);
        const int ftile = f / 128;
        const size_t e = (size_t)f * W + 8 * cg;
        if (cg * 8 == g.dv) {
            // z atom: column 0 holds sigma z, column 1 sigma itself (its
            // accumulator column is sigma times the row sum of the query
            // features, for the range check), columns 2..15 (the rest of the
            // N = 80 operand) zero
            float sum = 0.f;
            for (int gi = 0; gi < upto; ++gi) sum += st[gi * per + e] * scale[gi * g.n_ft + ftile];
            uint8_t *za = img + (size_t)nvb * g.r * 128;
            const uint32_t lo = __half_as_ushort(__float2half_rn(sum * sigma)) |
                                ((uint32_t)__half_as_ushort(__float2half_rn(sigma)) << 16);
            *reinterpret_cast<uint4 *>(za + sw128_offset(f, 0)) = make_uint4(lo, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(za + sw128_offset(f, 8)) = make_uint4(0u, 0u, 0u, 0u);
            continue;
        }
        float sum[8] = {};
        for (int gi = 0; gi < upto; ++gi) {
            const float sc = scale[gi * g.n_ft + ftile];
            const float *src = st + gi * per + e;
#pragma unroll
            for (int i = 0; i < 8; ++i) sum[i] = fmaf(src[i], sc, sum[i]);
        }
        const int c0 = 8 * cg;
        *reinterpret_cast<uint4 *>(img + (size_t)(c0 / 64) * g.r * 128 + sw128_offset(f, c0 % 64)) =
            make_uint4(pack_half2(sum[0] * sigma, sum[1] * sigma), pack_half2(sum[2] * sigma, sum[3] * sigma),
                       pack_half2(sum[4] * sigma, sum[5] * sigma), pack_half2(sum[6] * sigma, sum[7] * sigma));
    }
}

// ---------------------------------------------------------------------------
// tc_causal: the chunked causal scan, warp-specialised.
// Grid (segments, dv tiles, heads); 544 threads:
//   warp 0, lane 0  -- issues every TMA copy and tcgen05 MMA in order, waiting
//                      on mbarriers for the buffers it reuses;
//   warps 1..16     -- the epilogue group (512 threads, named barrier 1); warp
//                      w serves TMEM lane quarter w % 4 and column quarter
//                      (w - 1) / 4.
// Per chunk the tensor core runs: P_K = K W^T and P_Q = Q W^T (N = all
// projections); one N = 208 MMA with A = phi(Q) from TMEM against the rows
// KB = [phi(K); sigma S^T; sigma z^T] -> [A | phi_Q sigma S | phi_Q sigma z];
// S += phi(K)^T [V | 1] (N = 80) per 128 features; and [A_m V | A_m 1]
// (N = 80), A_m the masked, row-scaled A from TMEM.  The epilogue turns
// projections into features, the state into its fp16 rows of KB, A into A_m
// and the accumulators into out, staged for a TMA store.  P_Q is
// issued as soon as the epilogue holds P_K in registers, so the tensor core
// computes it while the key features are formed; the state rows of the next
// chunk are written while the tensor core computes its P_K.
// ---------------------------------------------------------------------------
constexpr int kCausalThreads = 32 + kEpi;
constexpr int kKbRows = 208;                     // phi_K 128 | sigma S^T 64 | sigma z 1 | ones 1 | pad 14
constexpr uint32_t kKbBlk = kKbRows * 128;       // one 64-feature block of the KB operand
constexpr int kKbS = 128, kKbZ = 192, kKbOne = 193;   // first rows of sigma S^T, sigma z, ones
// small-area float offsets of the barriers, TMEM slot, abort flag; total size
constexpr int kCausalBars = 1696, kCausalTslot = 1728, kCausalAbort = 1730, kCausalSmall = 1736;
static_assert(kCausalBars + 2 * 15 <= kCausalTslot, "the scan's mbarriers overlap the TMEM slot");
// r split: each row of a CTA's partial result travels as 68 floats (64 num,
// den, log2 scale, row sum of the query features, pad)
constexpr int kPartFloats = 68;

// 16 output values of one row (columns c0 .. c0 + 15) into a 128B-swizzled
// [128][64] bf16 staging block
__device__ __forceinline__ void stage_bf16_16(uint8_t *blk, int row, int c0, const float (&o)[16]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(o[8 * h + 2 * i], o[8 * h + 2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&b);
        }
        *reinterpret_cast<uint4 *>(blk + sw128_offset(row, c0 + 8 * h)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

struct CausalArgs {
    Geo g;                         // this CTA's features (one 128-feature slice in tc_causal_split)
    int H, L, seg_len, nseg;
    int rs;                        // CTAs per cluster splitting the features (1: no split)
    int nft_full, r_full;          // feature tiles and features of the whole head
    size_t w_head_bytes;           // bytes of one head's W image
    const uint8_t *omg;            // MN-major W images
    const float *s_in, *meta_in;   // [BH][nseg][r][dv+1], [BH][nseg][4] (segment 0 unused)
    const float *state, *meta;     // piece states [BH][nstate][r][dv+1], [BH][nstate][n_ft][4]
    int nstate, pps, direct;       // pps pieces per segment; direct: combine the earlier pieces here
    int out_bf16;                  // out in bf16 (one [128][64] staging block) instead of fp32
    int *status;
    void *out;                     // tc_causal_split: out [BH][L][dv] (fp32 or bf16), stored directly
    int nslots;                    // tc_causal_split: receive slots (2: no slot-free handshake)
    uint32_t o_w, o_x, o_v, o_kb, o_small, o_recv, o_stage, tmem_cols;
};

// TMEM columns: P [0, 256) | phi_Q packed [0, r/2) | A_m packed [0, 64) |
// [A_m V | A_m 1] [64, 144) | [A | phi_Q S | phi_Q z] [128, 336) | state
// tiles [352, 512), 80 columns each (dv values, then z)
constexpr int kColP = 0, kColB = 0, kColDI = 64, kColBig = 128, kColDX = 256, kColDD = 320,
              kColS = 352, kSStride = 80;

// 8 fp16 features (one 16-byte chunk) of a key row into the KB operand
__device__ __forceinline__ void kb_store8(uint8_t *kb, int row, int f, const float *v) {
    uint4 u = make_uint4(pack_half2(v[0], v[1]), pack_half2(v[2], v[3]), pack_half2(v[4], v[5]),
                         pack_half2(v[6], v[7]));
    *reinterpret_cast<uint4 *>(kb + (size_t)(f >> 6) * kKbBlk + sw128_offset(row, f & 63)) = u;
}

// NC = projection columns per epilogue thread (a quarter of the projections),
// MAP the feature map, OB16 out stored as bf16
template <int NC, int MAP, bool OB16>
__device__ void causal_body(const CausalArgs &a, uint8_t *sm, uint32_t tmem,
                            const CUtensorMap *tm_q, const CUtensorMap *tm_k,
                            const CUtensorMap *tm_v, const CUtensorMap *tm_out) {
    const Geo &g = a.g;
    const int seg = blockIdx.x, dvt = blockIdx.y, bh = blockIdx.z, head = bh % a.H;
    const int t_begin = seg * a.seg_len, t_end = min(a.L, t_begin + a.seg_len);
    const int nchunk = (t_end - t_begin + kC - 1) / kC;
    const int nd = g.d / 64, nft = g.n_ft, ft0 = 0, nft_full = a.nft_full;
    const uint32_t xb = (uint32_t)kC * g.d * 2;
    uint8_t *w = sm + a.o_w, *xq = sm + a.o_x, *xk = xq + xb, *xv = sm + a.o_v, *kb = sm + a.o_kb;
    float *small = reinterpret_cast<float *>(sm + a.o_small);
    float *nk = small;             // [128] half key norms (log2 units)
    float *part = small + 128;     // [4][128] query row max
    float *part2 = small + 640;    // [4][128] intra-chunk row max
    float *part3 = small + 1152;   // [4][128] key sums of squares
    float *red = small + 1664;     // [32]
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + kCausalBars);
    uint64_t *bar_w = &bars[0], *bar_x = &bars[1], *bar_v = &bars[2], *bar_pk = &bars[3],
             *bar_pq = &bars[4], *bar_a = &bars[5], *bar_av = &bars[6], *bar_st = &bars[13],
             *bar_in = &bars[14];
    uint64_t *e_x = &bars[7], *e_pk = &bars[8], *e_q = &bars[9], *e_v = &bars[10],
             *e_b = &bars[11], *e_out = &bars[12];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abortp = reinterpret_cast<volatile int *>(small + kCausalAbort);
    bool alive = true;

    if (warp == 0) {
        // ======================= control thread =======================
        if (lane == 0) {
            const uint32_t w_s = smem_u32(w), xq_s = smem_u32(xq), xk_s = smem_u32(xk),
                           v_s = smem_u32(xv), kb_s = smem_u32(kb);
            const uint32_t wbytes = (uint32_t)g.nproj * g.d * 2;
            auto load_x = [&](int c) {
                mbar_arrive_expect_tx(bar_x, 2 * xb);
                for (int b = 0; b < nd; ++b) {
                    tma_load_3d(xq + b * kBlk, tm_q, bar_x, 64 * b, t_begin + c * kC, bh);
                    tma_load_3d(xk + b * kBlk, tm_k, bar_x, 64 * b, t_begin + c * kC, bh);
                }
            };
            auto load_v = [&](int c) {
                mbar_arrive_expect_tx(bar_v, kBlk);
                tma_load_3d(xv, tm_v, bar_v, 64 * dvt, t_begin + c * kC, bh);
            };
            // P = X W^T over all projections (W MN-major: atoms of 64 projections)
            auto issue_proj = [&](uint32_t x_s) {
                const uint32_t idesc = idesc_f16(128, g.nproj, 0, 1);
                for (int kk = 0; kk < g.d / 16; ++kk)
                    mma_f16(tmem + kColP, smem_desc(x_s + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024),
                            smem_desc(w_s + kk * 2048, (uint32_t)g.d * 128, 1024), idesc, kk > 0);
            };
            if (nchunk > 0) {
                load_x(0);
                load_v(0);
            }
            // the W image (and the state of the earlier segments) come from
            // the kernels before this one
            grid_dep_wait();
            if (nchunk > 0) {
                mbar_arrive_expect_tx(bar_w, wbytes);
                bulk_load(w, a.omg + (size_t)head * a.w_head_bytes, wbytes, bar_w);
                alive = ewait(bar_w, 0, abortp);
            }
            for (int c = 0; c < nchunk && alive; ++c) {
                const uint32_t ph = c & 1;
                if (c == 0) {
                    if (!(alive = ewait(e_x, 0, abortp))) break;
                    tc_fence_after();
                    issue_proj(xk_s);
                    mma_commit(bar_pk);
                }
                // P_Q as soon as the epilogue holds P_K in registers
                if (!(alive = ewait(e_pk, ph, abortp))) break;
                tc_fence_after();
                issue_proj(xq_s);
                mma_commit(bar_pq);
                if (!(alive = ewait(bar_pq, ph, abortp))) break;
                if (c + 1 < nchunk) load_x(c + 1);
                // [A | phi_Q sigma S | phi_Q sigma z] = phi_Q KB^T once phi_Q,
                // phi_K and the state rows are in place
                if (!(alive = ewait(e_q, ph, abortp))) break;
                tc_fence_after();
                {
                    const uint32_t idesc = idesc_f16(128, kKbRows, 0, 0);
                    for (int kk = 0; kk < g.r / 16; ++kk)
                        mma_f16_ts(tmem + kColBig, tmem + 8 * kk,
                                   smem_desc(kb_s + (kk >> 2) * kKbBlk + (kk & 3) * 32, 16, 1024), idesc, kk > 0);
                }
                mma_commit(bar_a);
                // S += phi_K^T [V | 1] as soon as V is converted: it runs while
                // the epilogue masks and scales the intra-chunk matrix
                if (!(alive = ewait(e_v, ph, abortp))) break;
                tc_fence_after();
                {
                    const uint32_t ids = idesc_f16(128, 80, 1, 1);
                    for (int t = 0; t < nft; ++t)
                        for (int kk = 0; kk < kC / 16; ++kk)
                            mma_f16(tmem + kColS + t * kSStride,
                                    smem_desc(kb_s + (2 * t) * kKbBlk + kk * 2048, kKbBlk, 1024),
                                    smem_desc(v_s + kk * 2048, kBlk, 1024), ids, 1);
                }
                // [A_m V | A_m 1]
                if (!(alive = ewait(e_b, ph, abortp))) break;
                tc_fence_after();
                {
                    const uint32_t idv = idesc_f16(128, 80, 0, 1);
                    for (int kk = 0; kk < kC / 16; ++kk)
                        mma_f16_ts(tmem + kColDI, tmem + kColB + 8 * kk, smem_desc(v_s + kk * 2048, kBlk, 1024), idv, kk > 0);
                    mma_commit(bar_av);   // covers the state update issued before it
                }
                // the epilogue has staged out (fp32, two [128][32] halves in KB
                // rows 0..127 of blocks 0 and 1): store it, and once the store
                // has read the staging, the next chunk's key projection
                if (!(alive = ewait(e_out, ph, abortp))) break;
                tma_store_3d(tm_out, kb, 64 * dvt, t_begin + c * kC, bh);
                if (!OB16) tma_store_3d(tm_out, kb + kKbBlk, 64 * dvt + 32, t_begin + c * kC, bh);
                bulk_commit();
                if (c + 1 < nchunk) {
                    if (!(alive = ewait(e_x, (c + 1) & 1, abortp))) break;
                    tc_fence_after();
                    issue_proj(xk_s);
                    mma_commit(bar_pk);
                    if (!(alive = ewait(bar_av, ph, abortp))) break;
                    load_v(c + 1);
                    // the staging rows are phi_K rows again once the store has read them
                    bulk_wait_read0();
                    mbar_arrive(bar_st);
                }
            }
            bulk_wait0();
            if (!alive) set_status(a.status, FAVOR_ERR_TIMEOUT);
        }
        return;
    }
    // ======================= epilogue group =======================
    const int e = threadIdx.x - 32, ew = e >> 5;
    const int q = (ew + 1) & 3, j = ew >> 2;
    const int row = q * 32 + lane;
    float R = MAP == FAVOR_MAP_POSITIVE ? -INFINITY : 0.f, zmax = 0.f, vmax = 0.f;
    float s0[16], s1[16], z0 = 0.f, z1 = 0.f;   // this thread's part of the initial state
#pragma unroll
    for (int i = 0; i < 16; ++i) s0[i] = s1[i] = 0.f;
    // sigma S^T and sigma z -> KB rows kKbS.. and kKbZ, sigma a power of two
    // with sigma * (bound on max |S| and max z) <= kSigmaTarget.  alpha != 1
    // first rescales the state in TMEM (the key reference has moved).
    float sigma = 1.f;
    auto state_rows = [&](float alpha) {
        const float bound = zmax * fmaxf(vmax, 1.f);
        sigma = bound > 0.f ? pow2_scale_14(bound) : 1.f;
        const uint32_t kb_s = smem_u32(kb);
        for (int t = 0; t < nft; ++t) {
            const uint32_t col = kColS + t * kSStride;
            if (alpha != 1.f) {
                float s0[16], z0 = 0.f;
                tmem_ld16(tm_addr(tmem, q, col + 16 * j), s0);
                if (j == 0) tmem_ld1(tm_addr(tmem, q, col + 64), z0);
                tmem_ld_wait();
                uint32_t u[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(s0[i] * alpha);
                tmem_st16(tm_addr(tmem, q, col + 16 * j), u);
                if (j == 0) tmem_st1(tm_addr(tmem, q, col + 64), z0 * alpha);
                tmem_st_wait();
            }
            // this warp's 32 features x 16 value columns as four 16-lane x
            // 8-column fragments [h][g], stored transposed (rows = value
            // columns, 8 features per 16-byte chunk) by two stmatrix
            float a4[4][4], z0 = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int g = 0; g < 2; ++g)
                    tmem_ld_16x256b(tm_addr(tmem, q, col + 16 * j + 8 * g) + ((uint32_t)(16 * h) << 16), a4[2 * h + g]);
            if (j == 0) tmem_ld1(tm_addr(tmem, q, col + 64), z0);
            tmem_ld_wait();
            const int mi = lane >> 3;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int f = t * 128 + 32 * q + 16 * h + 8 * (mi & 1);
                const int rr = kKbS + 16 * j + 8 * (mi >> 1) + (lane & 7);
                const uint32_t addr = kb_s + (uint32_t)(f >> 6) * kKbBlk + (uint32_t)rr * 128u +
                                      ((((uint32_t)(f & 63) >> 3) ^ ((uint32_t)rr & 7u)) << 4);
                const float(&lo)[4] = a4[2 * h], (&hi)[4] = a4[2 * h + 1];
                stmatrix_x4_trans(addr, pack_half2(lo[0] * sigma, lo[1] * sigma), pack_half2(lo[2] * sigma, lo[3] * sigma),
                                  pack_half2(hi[0] * sigma, hi[1] * sigma), pack_half2(hi[2] * sigma, hi[3] * sigma));
            }
            if (j == 0) {
                const int f = t * 128 + row;
                *reinterpret_cast<__half *>(kb + (size_t)(f >> 6) * kKbBlk + sw128_offset(kKbZ, f & 63)) =
                    __float2half_rn(z0 * sigma);
            }
        }
    };
    auto convert_x = [&](int c) -> bool {
        const bool ok_x = ewait(bar_x, c & 1, abortp);
        float am, am2;
        convert_tile_512<false, true>(xq, nd, e, am);
        const float ss = convert_tile_512<true, true>(xk, nd, e, am2);
        if (fmaxf(am, am2) > kMaxOperand) flag_range(a.status);
        part3[(e >> 7) * 128 + (e & 127)] = ss;
        group_sync(kEpi);
        if (e < 128) nk[e] = 0.5f * kLog2e * ((part3[e] + part3[128 + e]) + (part3[256 + e] + part3[384 + e]));
        fence_async_smem();
        mbar_arrive(e_x);
        return ok_x;
    };
    // X(0) is the caller's data: convert it while the kernels before this
    // one finish; the state of the earlier segments is theirs
    if (nchunk > 0) alive = convert_x(0);
    grid_dep_wait();
    // The states of the earlier segments come through shared memory: bulk
    // copies of this CTA's state rows [nft x 128][dv + 1] (all of them, or
    // 128 or 64 at a time, as the KB area holds them) into the KB area, which
    // the scan takes over only after this; each thread then reads 16 values
    // of its row (rows 65 or 129 words apart fall on different banks)
    // instead of 16 scalar loads from global memory.
    const uint32_t row_floats = (uint32_t)g.dv + 1;
    const int span = nft * 128;
    const int kb_rows = (int)((uint32_t)(g.r / 64) * kKbBlk / (row_floats * 4u));
    const int unit = span <= kb_rows ? span : (128 <= kb_rows ? 128 : 64);
    float *stg = reinterpret_cast<float *>(kb);
    int sphase = 0;
    bool staged = false;
    auto take = [&](int lr, float (&sv)[16], float &zv, float sc) {
        const float *rp = stg + (size_t)lr * row_floats;
#pragma unroll
        for (int i = 0; i < 16; ++i) sv[i] += rp[64 * dvt + 16 * j + i] * sc;
        if (j == 0) zv += rp[g.dv] * sc;
    };
    // src: row 0 of this CTA's first feature tile; rows of tile t scaled by sc_t
    auto take_span = [&](const float *src, float sc0, float sc1) {
        for (int u = 0; u < span; u += unit) {
            if (staged) group_sync(kEpi);   // the previous staging has been read
            if (e == 0) {
                mbar_arrive_expect_tx(bar_in, (uint32_t)unit * row_floats * 4u);
                bulk_load(stg, src + (size_t)u * row_floats, (uint32_t)unit * row_floats * 4u, bar_in);
            }
            alive &= ewait(bar_in, sphase & 1, abortp);
            ++sphase;
            staged = true;
            if (row >= u && row < u + unit) take(row - u, s0, z0, sc0);
            if (nft == 2 && 128 + row >= u && 128 + row < u + unit) take(128 + row - u, s1, z1, sc1);
        }
    };
    if (seg > 0 && a.direct) {
        // the state after segments 0 .. seg-1 (pieces 0 .. seg pps - 1),
        // combined here at the largest of their key references (few segments:
        // no separate combine pass)
        const int npin = seg * a.pps;
        // [g][tile][R, max z, max|v|, max|S|]; this CTA's tiles ft0 .. ft0 + nft - 1
        const float *meta = a.meta + (size_t)bh * a.nstate * nft_full * 4 + (size_t)ft0 * 4;
        float Rs = -INFINITY;
        for (int gi = 0; gi < npin; ++gi)
            for (int t = 0; t < nft; ++t) {
                Rs = fmaxf(Rs, meta[(gi * nft_full + t) * 4]);
                vmax = fmaxf(vmax, meta[(gi * nft_full + t) * 4 + 2]);
            }
        auto scale = [&](int gi, int t) -> float {
            if (MAP != FAVOR_MAP_POSITIVE) return 1.f;
            const float Rg = meta[(gi * nft_full + t) * 4];
            return (Rg == -INFINITY || Rs == -INFINITY) ? 0.f : ex2(Rg - Rs);
        };
        for (int gi = 0; gi < npin; ++gi) {
            float zt = 0.f;
            for (int t = 0; t < nft; ++t) zt = fmaxf(zt, meta[(gi * nft_full + t) * 4 + 1] * scale(gi, t));
            zmax += zt;
        }
        if (MAP == FAVOR_MAP_POSITIVE) R = Rs;
        const size_t per = (size_t)a.r_full * (g.dv + 1);
        for (int gi = 0; gi < npin; ++gi) {
            const float *st = a.state + ((size_t)bh * a.nstate + gi) * per + (size_t)ft0 * 128 * row_floats;
            take_span(st, scale(gi, 0), nft == 2 ? scale(gi, 1) : 0.f);
        }
    } else if (seg > 0) {
        const float *m = a.meta_in + ((size_t)bh * a.nseg + seg) * 4;
        R = m[0];
        zmax = m[1];
        vmax = m[2];
        take_span(a.s_in + (((size_t)bh * a.nseg + seg) * a.r_full + (size_t)ft0 * 128) * row_floats, 1.f, 1.f);
    }
    // the KB area is the scan's from here: every staged row has been read
    if (staged) group_sync(kEpi);
    // the ones row (its accumulator column is the row sum of the query
    // features, for the range check) and the pad rows after it (they feed
    // accumulator columns never read)
    for (int i = e; i < (g.r / 64) * 15 * 8; i += kEpi) {
        const int blk = i / 120, rr = kKbOne + (i % 120) / 8, ch = i % 8;
        const uint32_t one = rr == kKbOne ? 0x3C003C00u : 0u;
        *reinterpret_cast<uint4 *>(kb + (size_t)blk * kKbBlk + rr * 128 + ch * 16) = make_uint4(one, one, one, one);
    }
    fence_async_smem();
    // initial state into TMEM: tile t, lanes = features, 16 value columns per thread
    {
        uint32_t u[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(s0[i]);
        tmem_st16(tm_addr(tmem, q, kColS + 16 * j), u);
        if (j == 0) tmem_st1(tm_addr(tmem, q, kColS + 64), z0);
        if (nft == 2) {
#pragma unroll
            for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(s1[i]);
            tmem_st16(tm_addr(tmem, q, kColS + kSStride + 16 * j), u);
            if (j == 0) tmem_st1(tm_addr(tmem, q, kColS + kSStride + 64), z1);
        }
        tmem_st_wait();
    }
    state_rows(1.f);
    for (int c = 0; c < nchunk; ++c) {
        const uint32_t ph = c & 1;
        const int tc0 = t_begin + c * kC;
        const int valid = min(kC, t_end - tc0);
        const bool ok = row < valid;
        // ---------------- key features -> KB rows 0..127 ----------------
        alive &= ewait(bar_pk, ph, abortp);
        tc_fence_after();
        const uint32_t pcol = tm_addr(tmem, q, kColP + NC * j);
        float pv[NC];
#pragma unroll
        for (int b = 0; b < NC / 16; ++b) {
            float t16[16];
            tmem_ld16(pcol + 16 * b, t16);
#pragma unroll
            for (int i = 0; i < 16; ++i) pv[16 * b + i] = t16[i];
        }
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(e_pk);   // P_K is in registers: P_Q may overwrite it
        // KB rows 0..127 held the previous chunk's output staging
        if (c > 0) alive &= ewait(bar_st, (c - 1) & 1, abortp);
        const float nkr = nk[row];
        float mf = 0.f, moved = 1.f;   // moved: state rescale when the key reference moves
        if constexpr (MAP == FAVOR_MAP_POSITIVE) {
            const float mx = max_of(pv);
            // a key whose largest feature would pass e^(shift + slack) at the
            // current reference (always so before the first key) moves the
            // reference to it; the state so far is rescaled below
            if (group_or(ok && mx - nkr - R > kLog2MaxFeature, kEpi)) {
                const float Rn = grp_max(ok ? mx - nkr : -INFINITY, red, ew) - kShift;
                if (R != -INFINITY) moved = ex2(R - Rn);
                R = Rn;
            }
            // rows past the end take an infinite offset: their features are 0
            const float off = ok ? nkr + R : INFINITY;
            mf = ex2(mx - off);
#pragma unroll
            for (int b = 0; b < NC / 8; ++b) {
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = ex2(pv[8 * b + i] - off);
                kb_store8(kb, row, NC * j + 8 * b, v);
            }
        } else if constexpr (MAP == FAVOR_MAP_TRIG) {
            // projection p -> features 128 (p / 64) + p % 64 (sin) and that + 64
            // (cos): each 128-feature tile holds the sin and cos of 64 projections
            const int fs = 128 * ((NC * j) / 64) + (NC * j) % 64;
#pragma unroll
            for (int b = 0; b < NC / 8; ++b) {
                float s8[8], c8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (ok) sincos_reduced(pv[8 * b + i], s8[i], c8[i]);
                    else s8[i] = c8[i] = 0.f;
                    mf = fmaxf(mf, fmaxf(fabsf(s8[i]), fabsf(c8[i])));
                }
                kb_store8(kb, row, fs + 8 * b, s8);
                kb_store8(kb, row, fs + 64 + 8 * b, c8);
            }
        } else {
#pragma unroll
            for (int b = 0; b < NC / 8; ++b) {
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    v[i] = ok ? elu1(pv[8 * b + i]) : 0.f;
                    mf = fmaxf(mf, v[i]);
                }
                kb_store8(kb, row, NC * j + 8 * b, v);
            }
        }
        if (moved != 1.f) {
            // the state so far and its rows in KB move to the new reference
            zmax *= moved;
            state_rows(moved);
        }
        // ---------------- query features -> phi_Q in TMEM [0, r/2) ----------------
        alive &= ewait(bar_pq, ph, abortp);
        tc_fence_after();
#pragma unroll
        for (int b = 0; b < NC / 16; ++b) {
            float t16[16];
            tmem_ld16(pcol + 16 * b, t16);
#pragma unroll
            for (int i = 0; i < 16; ++i) pv[16 * b + i] = t16[i];
        }
        tmem_ld_wait();
        float qoff = 0.f;
        if constexpr (MAP == FAVOR_MAP_POSITIVE) part[j * 128 + row] = max_of(pv);
        tc_fence_before();
        group_sync(kEpi);   // every projection column read: phi_Q may now overwrite them
        tc_fence_after();

        if constexpr (MAP == FAVOR_MAP_POSITIVE) {
            qoff = fmaxf(fmaxf(part[row], part[128 + row]), fmaxf(part[256 + row], part[384 + row])) - kShift;
#pragma unroll
            for (int b = 0; b < NC / 32; ++b) {
                uint32_t o[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    o[i] = pack_half2(ex2(pv[32 * b + 2 * i] - qoff), ex2(pv[32 * b + 2 * i + 1] - qoff));
                tmem_st16(tm_addr(tmem, q, (NC * j + 32 * b) / 2), o);
            }
        } else if constexpr (MAP == FAVOR_MAP_TRIG) {
            // same feature order as the keys; 16 projections give 8 packed
            // columns of sin and 8 of cos
            const int fs = 128 * ((NC * j) / 64) + (NC * j) % 64;
#pragma unroll
            for (int b = 0; b < NC / 16; ++b) {
                uint32_t os[8], oc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float s0, c0, s1, c1;
                    sincos_reduced(pv[16 * b + 2 * i], s0, c0);
                    sincos_reduced(pv[16 * b + 2 * i + 1], s1, c1);
                    os[i] = pack_half2(s0, s1);
                    oc[i] = pack_half2(c0, c1);
                }
                tmem_st8(tm_addr(tmem, q, (fs + 16 * b) / 2), os);
                tmem_st8(tm_addr(tmem, q, (fs + 64 + 16 * b) / 2), oc);
            }
        } else {
#pragma unroll
            for (int b = 0; b < NC / 32; ++b) {
                uint32_t o[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    o[i] = pack_half2(elu1(pv[32 * b + 2 * i]), elu1(pv[32 * b + 2 * i + 1]));
                tmem_st16(tm_addr(tmem, q, (NC * j + 32 * b) / 2), o);
            }
        }
        tmem_st_wait();
        fence_async_smem();   // KB rows (features, state) for the tensor core
        tc_fence_before();
        mbar_arrive(e_q);
        // ---------------- V -> fp16, running max |v| ----------------
        alive &= ewait(bar_v, ph, abortp);
        {
            float am;
            convert_tile_512<false, true>(xv, 1, e, am);
            if (am > kMaxOperand) flag_range(a.status);
            fence_async_smem();
            mbar_arrive(e_v);
            // warp partials of max |v| and of the key mass (sum over keys of the
            // largest feature, the bound on the growth of z); the group combines
            // them after the barrier of the next Q, K conversion
            float ms = mf;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
                ms += __shfl_xor_sync(0xffffffffu, ms, o);
            }
            if (lane == 0) {
                red[ew] = am;
                red[16 + ew] = ms;
            }
        }
        // ---------------- next chunk's Q, K (while the tensor core runs the merged MMA) ----------------
        if (c + 1 < nchunk) {
            alive &= convert_x(c + 1);   // its group barrier publishes red
            float vm = red[0], ms = 0.f;
#pragma unroll
            for (int i = 0; i < kEpi / 32; ++i) {
                vm = fmaxf(vm, red[i]);
                ms += red[16 + i];
            }
            vmax = fmaxf(vmax, vm);
            zmax += ms;
        }
        // ---------------- intra-chunk matrix -> masked, row-scaled, TMEM ----------------
        alive &= ewait(bar_a, ph, abortp);
        tc_fence_after();
        float av[32];
        const int limit = min(row, valid - 1) - 32 * j;   // keys j' <= limit (local index)
        float rm = 0.f;
        if (limit < 0) {                 // this quarter lies entirely above the diagonal
#pragma unroll
            for (int i = 0; i < 32; ++i) av[i] = 0.f;
        } else {
            tmem_ld32(tm_addr(tmem, q, kColBig + 32 * j), av);
            tmem_ld_wait();
            if (limit < 31) {
#pragma unroll
                for (int i = 0; i < 32; ++i) av[i] = i <= limit ? av[i] : 0.f;
            }
            {
                float aa[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) aa[i] = fabsf(av[i]);
                rm = max_of(aa);
            }
        }
        part2[j * 128 + row] = rm;
        group_sync(kEpi);
        const float rmax = fmaxf(fmaxf(part2[row], part2[128 + row]), fmaxf(part2[256 + row], part2[384 + row]));
        const float rho = rmax > 0.f ? pow2_inv_floor(rmax) : 1.f;
        {
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = pack_half2(av[2 * i] * rho, av[2 * i + 1] * rho);
            tmem_st16(tm_addr(tmem, q, kColB + 16 * j), o);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(e_b);
        // ---------------- output ----------------
        alive &= ewait(bar_av, ph, abortp);
        tc_fence_after();
        {
            float di[16], dx[16], ddi, ddx, qsum = 0.f;
            tmem_ld16(tm_addr(tmem, q, kColDI + 16 * j), di);
            tmem_ld16(tm_addr(tmem, q, kColDX + 16 * j), dx);
            tmem_ld1(tm_addr(tmem, q, kColDI + 64), ddi);
            tmem_ld1(tm_addr(tmem, q, kColDD), ddx);
            if (j == 0) tmem_ld1(tm_addr(tmem, q, kColDD + 1), qsum);
            tmem_ld_wait();
            tc_fence_before();
            const float is = pow2_inv_floor(sigma), ir = pow2_inv_floor(rho);   // exact: powers of two
            float ov[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = fmaf(di[i], ir, dx[i] * is);
            float den = fmaf(ddi, ir, ddx * is);
            const float id = __fdividef(1.f, den);
            // the range check: the denominator against the features' fp16
            // floor (keys so far x the row sum of the query features x the
            // flush level, with a 2^10 margin)
            if (MAP == FAVOR_MAP_POSITIVE && j == 0 && ok && den < (float)(tc0 + row + 1) * qsum * kRangeFloor)
                flag_range(a.status);
            {
                if constexpr (OB16) {
                    // output columns 16 j .. 16 j + 15 -> the bf16 staging block
                    // (phi_K rows of KB block 0, free since the state update)
                    float o[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] = ov[i] * id;
                    stage_bf16_16(kb, row, 16 * j, o);
                } else {
                    // output columns 16 j .. 16 j + 15 -> staging half (16 j) / 32 (the
                    // phi_K rows of KB block 0 or 1, free since the state update), 128B
                    // swizzle in chunks of 4 floats
                    uint8_t *half = kb + (size_t)((16 * j) >> 5) * kKbBlk;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int col = (16 * j + 4 * cc) & 31;
                        const int p = (col >> 2) ^ (row & 7);
                        *reinterpret_cast<float4 *>(half + row * 128 + p * 16) =
                            make_float4(ov[4 * cc] * id, ov[4 * cc + 1] * id, ov[4 * cc + 2] * id, ov[4 * cc + 3] * id);
                    }
                }
            }
            fence_async_smem();
            mbar_arrive(e_out);
        }
        // ---------------- state rows of the next chunk (during its P_K) ----------------
        if (c + 1 < nchunk) state_rows(1.f);
    }
    if (!alive) set_status(a.status, FAVOR_ERR_TIMEOUT);
}

// OB16: out stored as bf16 (a kernel of its own, so that the fp32 kernel's
// registers are allocated for the fp32 epilogue alone)
template <bool OB16>
__global__ void __launch_bounds__(kCausalThreads, 1)
tc_causal(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
          const CausalArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *small = reinterpret_cast<float *>(sm + a.o_small);
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + kCausalBars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(small + kCausalTslot);
    volatile int *abortp = reinterpret_cast<volatile int *>(small + kCausalAbort);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        *abortp = 0;
        for (int i = 0; i < 7; ++i) mbar_init(&bars[i], 1);
        for (int i = 7; i < 13; ++i) mbar_init(&bars[i], kEpi);
        mbar_init(&bars[13], 1);
        mbar_init(&bars[14], 1);
        fence_mbar_init();
    }
    // ones atom after the V tile: the z column of S += phi_K^T [V | 1] and
    // the row sums of [A_m V | A_m 1]
    uint8_t *ones = sm + a.o_v + kBlk;
    for (int i = threadIdx.x; i < (int)(kBlk / 16); i += kCausalThreads)
        reinterpret_cast<uint4 *>(ones)[i] = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    if (warp == 0) tmem_alloc(tslot, a.tmem_cols);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int nc = a.g.nproj / 4;
    grid_dep_launch();
    if (a.g.map == FAVOR_MAP_POSITIVE) {
        if (nc == 64) causal_body<64, FAVOR_MAP_POSITIVE, OB16>(a, sm, tmem, &tm_q, &tm_k, &tm_v, &tm_out);
        else causal_body<32, FAVOR_MAP_POSITIVE, OB16>(a, sm, tmem, &tm_q, &tm_k, &tm_v, &tm_out);
    } else if (a.g.map == FAVOR_MAP_TRIG) {
        if (nc == 32) causal_body<32, FAVOR_MAP_TRIG, OB16>(a, sm, tmem, &tm_q, &tm_k, &tm_v, &tm_out);
        else causal_body<16, FAVOR_MAP_TRIG, OB16>(a, sm, tmem, &tm_q, &tm_k, &tm_v, &tm_out);
    } else {
        causal_body<32, FAVOR_MAP_ELU1, OB16>(a, sm, tmem, &tm_q, &tm_k, &tm_v, &tm_out);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, a.tmem_cols);
}

// ---------------------------------------------------------------------------
// tc_causal_split: the chunked causal scan of a head whose features are
// split over the rs CTAs of a cluster (rs = r / 128: one 128-feature slice
// each; rs = 1 would be a whole head of 128).  Each CTA scans its slice at
// its own key reference and query offsets; per chunk every CTA sends its
// partial numerators, denominators and log-scales for the rows another CTA
// finalises through distributed shared memory (st.async completing on the
// owner's mbarrier), and each owner rescales, sums, normalises and stores its
// rows.  With 128 features the projections, the query features, the
// intra-chunk matrix and the state leave TMEM room for a second chunk, so
// the scan is software-pipelined by one chunk: the tensor core projects
// chunk c + 1 and the epilogue forms its features while chunk c's masked
// product A_m [V | 1] runs and its output is reduced and stored.
//   control thread, per chunk c:  merged MMA (c) | P_K (c + 1) |
//     S += phi_K^T [V | 1] (c) | A_m [V | 1] (c) | P_Q (c + 1) | loads
//   epilogue, per chunk c:  masked, row-scaled A (c) | key features and
//     state rows (c + 1) | query features (c + 1) | partial output (c), sent
//     | phi_Q (c + 1) into TMEM | Q, K (c + 2) -> fp16 | output (c) gathered
//     and stored | V (c + 1) -> fp16
// TMEM: P [0, 128) | A_m [V | 1] at [128, 208), phi_Q (packed) there before
// it (the merged MMA has consumed phi_Q when A_m V overwrites it) | [A |
// phi_Q sigma S | phi_Q sigma z | query row sum] at [208, 416), A_m packed
// in place (keys 32 j .. 32 j + 31 in columns 208 + 32 j .. + 15) | the
// state [416, 496) (64 values, z).
// Shared memory: W slice, Q and K tiles, V tile + ones atom, KB (phi_K 128
// rows, sigma S^T 64, sigma z, ones) per 64 features, the small area, and one
// or two receive slots: per sender, the numerators [4 column quarters][rows
// 128 / rs][16] (each owner thread reads 64 contiguous bytes) and then
// [rows][den, log2 scale, query row sum, pad].  With two slots (by chunk
// parity) a sender never waits: it writes slot c % 2 only after it has
// received the owner's partials of chunk c - 1, which the owner sends after it
// has read slot c % 2 for chunk c - 2.  With one slot every owner warp tells
// the senders when it has read it.  The owners store their rows straight to
// global memory (64 contiguous bytes per thread).
// ---------------------------------------------------------------------------
constexpr int kPcP = 0, kPcAV = 128, kPcA = 208, kPcDX = 336, kPcDD = 400, kPcS = 416;
// small-area float offsets of the split scan
constexpr int kSpRedM = 1696, kSpRedV = 1728, kSpBars = 1760, kSpTslot = 1800, kSpAbort = 1802, kSpSmall = 1808;
constexpr int kSpNumBars = 18;
static_assert(kSpBars + 2 * kSpNumBars <= kSpTslot, "the split scan's mbarriers overlap the TMEM slot");

template <int NC, int MAP, bool OB16>
__device__ void split_body(const CausalArgs &a, uint8_t *sm, uint32_t tmem, const CUtensorMap *tm_q,
                           const CUtensorMap *tm_k, const CUtensorMap *tm_v, const CUtensorMap *tm_out) {
    const Geo &g = a.g;
    const int rs = a.rs, seg = blockIdx.x / rs, slice = blockIdx.x % rs;
    const int dvt = blockIdx.y, bh = blockIdx.z, head = bh % a.H;
    const int t_begin = seg * a.seg_len, t_end = min(a.L, t_begin + a.seg_len);
    const int nchunk = (t_end - t_begin + kC - 1) / kC;
    const int nd = g.d / 64, ft0 = slice, nft_full = a.nft_full;
    const int rpo = kC / rs;
    const uint32_t xb = (uint32_t)kC * g.d * 2;
    uint8_t *w = sm + a.o_w, *xq = sm + a.o_x, *xk = xq + xb, *xv = sm + a.o_v, *kb = sm + a.o_kb;
    float *small = reinterpret_cast<float *>(sm + a.o_small);
    float *nk = small;             // [128] half key norms (log2 units)
    float *part = small + 128;     // [4][128] query row max
    float *part2 = small + 640;    // [4][128] intra-chunk row max
    float *part3 = small + 1152;   // [4][128] key sums of squares
    float *red = small + 1664;     // [32] the vote
    float *redm = small + kSpRedM; // [2][16] key mass per warp, by chunk parity
    float *redv = small + kSpRedV; // [2][16] max |v| per warp, by chunk parity
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + kSpBars);
    uint64_t *b_w = &bars[0], *b_x = &bars[1], *b_v = &bars[2], *b_pk = &bars[3], *b_pq = &bars[4],
             *b_a = &bars[5], *b_s = &bars[6], *b_av = &bars[7];
    uint64_t *e_x = &bars[9], *e_pk = &bars[10], *e_q = &bars[11], *e_v = &bars[12], *e_b = &bars[13];
    uint64_t *bar_free = &bars[16], *bar_in = &bars[8];
    // receive slot s: its barrier, its numerators and its per-row scalars
    const int nslots = a.nslots;
    const size_t slot_floats = (size_t)(rs - 1) * rpo * kPartFloats;
    auto bar_recv = [&](int slot) { return &bars[slot ? 17 : 15]; };
    auto recv_num = [&](int slot, int sidx, int quarter, int lr) {
        return reinterpret_cast<float *>(sm + a.o_recv) + slot * slot_floats +
               ((size_t)(sidx * 4 + quarter) * rpo + lr) * 16;
    };
    auto recv_meta = [&](int slot, int sidx, int lr) {
        return reinterpret_cast<float *>(sm + a.o_recv) + slot * slot_floats + (size_t)(rs - 1) * rpo * 64 +
               ((size_t)sidx * rpo + lr) * 4;
    };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abortp = reinterpret_cast<volatile int *>(small + kSpAbort);
    bool alive = true;

    if (warp == 0) {
        // ======================= control thread =======================
        if (lane == 0) {
            const uint32_t w_s = smem_u32(w), xq_s = smem_u32(xq), xk_s = smem_u32(xk), v_s = smem_u32(xv),
                           kb_s = smem_u32(kb);
            const uint32_t wbytes = (uint32_t)g.nproj * g.d * 2;
            auto load_x = [&](int c) {
                mbar_arrive_expect_tx(b_x, 2 * xb);
                for (int b = 0; b < nd; ++b) {
                    tma_load_3d(xq + b * kBlk, tm_q, b_x, 64 * b, t_begin + c * kC, bh);
                    tma_load_3d(xk + b * kBlk, tm_k, b_x, 64 * b, t_begin + c * kC, bh);
                }
            };
            auto load_v = [&](int c) {
                mbar_arrive_expect_tx(b_v, kBlk);
                tma_load_3d(xv, tm_v, b_v, 64 * dvt, t_begin + c * kC, bh);
            };
            // P = X W^T (N = the slice's projections)
            auto proj = [&](uint32_t x_s) {
                const uint32_t idesc = idesc_f16(128, g.nproj, 0, 1);
                for (int kk = 0; kk < g.d / 16; ++kk)
                    mma_f16(tmem + kPcP, smem_desc(x_s + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024),
                            smem_desc(w_s + kk * 2048, (uint32_t)g.d * 128, 1024), idesc, kk > 0);
            };
            if (nchunk > 0) {
                load_x(0);
                load_v(0);
            }
            // the W image (and the state of the earlier segments) come from
            // the kernels before this one
            grid_dep_wait();
            if (nchunk > 0) {
                mbar_arrive_expect_tx(b_w, wbytes);
                bulk_load(w, a.omg + (size_t)head * a.w_head_bytes + (size_t)slice * wbytes, wbytes, b_w);
                alive = ewait(b_w, 0, abortp) && ewait(e_x, 0, abortp);
                if (alive) {
                    tc_fence_after();
                    proj(xk_s);
                    mma_commit(b_pk);
                    alive = ewait(e_pk, 0, abortp);
                }
                if (alive) {
                    tc_fence_after();
                    proj(xq_s);
                    mma_commit(b_pq);
                    alive = ewait(b_pq, 0, abortp);
                    if (alive && nchunk > 1) load_x(1);
                }
            }
            for (int c = 0; c < nchunk && alive; ++c) {
                const uint32_t ph = c & 1, ph1 = (c + 1) & 1;
                const bool more = c + 1 < nchunk;
                // [A | phi_Q sigma S | phi_Q sigma z | q sum] = phi_Q KB^T
                if (!(alive = ewait(e_q, ph, abortp))) break;
                tc_fence_after();
                {
                    const uint32_t idesc = idesc_f16(128, kKbRows, 0, 0);
                    for (int kk = 0; kk < g.r / 16; ++kk)
                        mma_f16_ts(tmem + kPcA, tmem + kPcAV + 8 * kk,
                                   smem_desc(kb_s + (kk >> 2) * kKbBlk + (kk & 3) * 32, 16, 1024), idesc, kk > 0);
                    mma_commit(b_a);
                }
                // the next chunk's key projection (P was read for chunk c's queries)
                if (more) {
                    if (!(alive = ewait(e_x, ph1, abortp))) break;
                    tc_fence_after();
                    proj(xk_s);
                    mma_commit(b_pk);
                }
                // S += phi_K^T [V | 1]
                if (!(alive = ewait(e_v, ph, abortp))) break;
                tc_fence_after();
                {
                    const uint32_t ids = idesc_f16(128, 80, 1, 1);
                    for (int kk = 0; kk < kC / 16; ++kk)
                        mma_f16(tmem + kPcS, smem_desc(kb_s + kk * 2048, kKbBlk, 1024),
                                smem_desc(v_s + kk * 2048, kBlk, 1024), ids, 1);
                    mma_commit(b_s);
                }
                // [A_m V | A_m 1], A_m packed in place in the A columns
                if (!(alive = ewait(e_b, ph, abortp))) break;
                tc_fence_after();
                {
                    const uint32_t idv = idesc_f16(128, 80, 0, 1);
                    for (int kk = 0; kk < kC / 16; ++kk)
                        mma_f16_ts(tmem + kPcAV, tmem + kPcA + 32 * (kk >> 1) + 8 * (kk & 1),
                                   smem_desc(v_s + kk * 2048, kBlk, 1024), idv, kk > 0);
                    mma_commit(b_av);
                }
                // the next chunk's query projection, then its Q, K tiles
                if (more) {
                    if (!(alive = ewait(e_pk, ph1, abortp))) break;
                    tc_fence_after();
                    proj(xq_s);
                    mma_commit(b_pq);
                    if (!(alive = ewait(b_pq, ph1, abortp))) break;
                    if (c + 2 < nchunk) load_x(c + 2);
                }
                // V is free once A_m V (and the state update before it) is done
                if (!(alive = ewait(b_av, ph, abortp))) break;
                if (more) load_v(c + 1);
            }

            if (!alive) set_status(a.status, FAVOR_ERR_TIMEOUT);
        }
        return;
    }
    // ======================= epilogue group =======================
    const int e = threadIdx.x - 32, ew = e >> 5;
    const int q = (ew + 1) & 3, j = ew >> 2;
    const int row = q * 32 + lane;
    float R = MAP == FAVOR_MAP_POSITIVE ? -INFINITY : 0.f, zmax = 0.f, vmax = 0.f, sigma = 1.f;
    float qoff_next = 0.f;                  // query row offset of the chunk whose features are held
    constexpr int NH = MAP == FAVOR_MAP_TRIG ? NC : NC / 2;
    uint32_t hq[NH];                        // that chunk's query features, packed fp16
    float s0[16], z0 = 0.f;                 // this thread's part of the initial state
#pragma unroll
    for (int i = 0; i < 16; ++i) s0[i] = 0.f;

    // sigma S^T and sigma z -> KB rows kKbS.. and kKbZ (sigma: a power of two
    // with sigma * (bound on max |S| and max z) <= kSigmaTarget); alpha != 1
    // first rescales the state in TMEM (the key reference has moved)
    auto state_rows = [&](float alpha) {
        const float bound = zmax * fmaxf(vmax, 1.f);
        sigma = bound > 0.f ? pow2_scale_14(bound) : 1.f;
        const uint32_t kb_s = smem_u32(kb);
        if (alpha != 1.f) {
            float t16[16], zz = 0.f;
            tmem_ld16(tm_addr(tmem, q, kPcS + 16 * j), t16);
            if (j == 0) tmem_ld1(tm_addr(tmem, q, kPcS + 64), zz);
            tmem_ld_wait();
            uint32_t u[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(t16[i] * alpha);
            tmem_st16(tm_addr(tmem, q, kPcS + 16 * j), u);
            if (j == 0) tmem_st1(tm_addr(tmem, q, kPcS + 64), zz * alpha);
            tmem_st_wait();
        }
        float a4[4][4], zz = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int g2 = 0; g2 < 2; ++g2)
                tmem_ld_16x256b(tm_addr(tmem, q, kPcS + 16 * j + 8 * g2) + ((uint32_t)(16 * h) << 16), a4[2 * h + g2]);
        if (j == 0) tmem_ld1(tm_addr(tmem, q, kPcS + 64), zz);
        tmem_ld_wait();
        const int mi = lane >> 3;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int f = 32 * q + 16 * h + 8 * (mi & 1);
            const int rr = kKbS + 16 * j + 8 * (mi >> 1) + (lane & 7);
            const uint32_t addr = kb_s + (uint32_t)(f >> 6) * kKbBlk + (uint32_t)rr * 128u +
                                  ((((uint32_t)(f & 63) >> 3) ^ ((uint32_t)rr & 7u)) << 4);
            const float(&lo)[4] = a4[2 * h], (&hi)[4] = a4[2 * h + 1];
            stmatrix_x4_trans(addr, pack_half2(lo[0] * sigma, lo[1] * sigma), pack_half2(lo[2] * sigma, lo[3] * sigma),
                              pack_half2(hi[0] * sigma, hi[1] * sigma), pack_half2(hi[2] * sigma, hi[3] * sigma));
        }
        if (j == 0)
            *reinterpret_cast<__half *>(kb + (size_t)(row >> 6) * kKbBlk + sw128_offset(kKbZ, row & 63)) =
                __float2half_rn(zz * sigma);
    };
    auto convert_x = [&](int c) -> bool {
        const bool ok_x = ewait(b_x, c & 1, abortp);
        float am, am2;
        convert_tile_512<false, true>(xq, nd, e, am);
        const float ss = convert_tile_512<true, true>(xk, nd, e, am2);
        if (fmaxf(am, am2) > kMaxOperand) flag_range(a.status);
        part3[(e >> 7) * 128 + (e & 127)] = ss;
        group_sync(kEpi);
        if (e < 128) nk[e] = 0.5f * kLog2e * ((part3[e] + part3[128 + e]) + (part3[256 + e] + part3[384 + e]));
        fence_async_smem();
        mbar_arrive(e_x);
        return ok_x;
    };
    // key features of chunk c -> KB rows 0..127 (after the vote on the key
    // reference); returns the factor the state so far moves by
    auto keys = [&](int c) -> float {
        const int valid = min(kC, t_end - (t_begin + c * kC));
        const bool ok = row < valid;
        alive &= ewait(b_pk, c & 1, abortp);
        tc_fence_after();
        float pv[NC];
        tmem_ld_cols<NC>(tm_addr(tmem, q, kPcP + NC * j), pv);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(e_pk);   // P_K is in registers: P_Q may overwrite it
        const float nkr = nk[row];
        float mf = 0.f, moved = 1.f;
        float off = 0.f;
        if constexpr (MAP == FAVOR_MAP_POSITIVE) {
            const float mx = max_of(pv);
            if (group_or(ok && mx - nkr - R > kLog2MaxFeature, kEpi)) {
                const float Rn = grp_max(ok ? mx - nkr : -INFINITY, red, ew) - kShift;
                if (R != -INFINITY) moved = ex2(R - Rn);
                R = Rn;
            }
            off = ok ? nkr + R : INFINITY;
            mf = ex2(mx - off);
        }
        // phi_K rows and the state are free once the update of chunk c - 1 is done
        if (c > 0) alive &= ewait(b_s, (c - 1) & 1, abortp);
        tc_fence_after();
        if constexpr (MAP == FAVOR_MAP_POSITIVE) {
#pragma unroll
            for (int b = 0; b < NC / 8; ++b) {
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = ex2(pv[8 * b + i] - off);
                kb_store8(kb, row, NC * j + 8 * b, v);
            }
        } else if constexpr (MAP == FAVOR_MAP_TRIG) {
            // projection p -> feature p (sin) and p + 64 (cos) of the slice
            const int fs = NC * j;
#pragma unroll
            for (int b = 0; b < NC / 8; ++b) {
                float s8[8], c8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (ok) sincos_reduced(pv[8 * b + i], s8[i], c8[i]);
                    else s8[i] = c8[i] = 0.f;
                    mf = fmaxf(mf, fmaxf(fabsf(s8[i]), fabsf(c8[i])));
                }
                kb_store8(kb, row, fs + 8 * b, s8);
                kb_store8(kb, row, fs + 64 + 8 * b, c8);
            }
        } else {
#pragma unroll
            for (int b = 0; b < NC / 8; ++b) {
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    v[i] = ok ? elu1(pv[8 * b + i]) : 0.f;
                    mf = fmaxf(mf, v[i]);
                }
                kb_store8(kb, row, NC * j + 8 * b, v);
            }
        }
        // warp partial of the key mass (sum over keys of the largest feature,
        // the bound on the growth of z), read after the next group barrier
        float ms = mf;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ms += __shfl_xor_sync(0xffffffffu, ms, o);
        if (lane == 0) redm[(c & 1) * 16 + ew] = ms;
        return moved;
    };
    // query features of chunk c -> registers (hq), its row offset -> qoff_next
    auto queries = [&](int c) {
        alive &= ewait(b_pq, c & 1, abortp);
        tc_fence_after();
        float pv[NC];
        tmem_ld_cols<NC>(tm_addr(tmem, q, kPcP + NC * j), pv);
        tmem_ld_wait();
        tc_fence_before();
        if constexpr (MAP == FAVOR_MAP_POSITIVE) {
            part[j * 128 + row] = max_of(pv);
            group_sync(kEpi);
            qoff_next = fmaxf(fmaxf(part[row], part[128 + row]), fmaxf(part[256 + row], part[384 + row])) - kShift;
#pragma unroll
            for (int i = 0; i < NC / 2; ++i) hq[i] = pack_half2(ex2(pv[2 * i] - qoff_next), ex2(pv[2 * i + 1] - qoff_next));
        } else if constexpr (MAP == FAVOR_MAP_TRIG) {
            // sines in hq[0, NC/2), cosines in hq[NC/2, NC)
#pragma unroll
            for (int i = 0; i < NC / 2; ++i) {
                float sa, ca, sb, cb;
                sincos_reduced(pv[2 * i], sa, ca);
                sincos_reduced(pv[2 * i + 1], sb, cb);
                hq[i] = pack_half2(sa, sb);
                hq[NC / 2 + i] = pack_half2(ca, cb);
            }
        } else {
#pragma unroll
            for (int i = 0; i < NC / 2; ++i) hq[i] = pack_half2(elu1(pv[2 * i]), elu1(pv[2 * i + 1]));
        }
    };
    // the held query features -> TMEM (the A_m V columns, read by the output
    // of the previous chunk first); then the merged MMA may start
    auto store_q = [&]() {
        group_sync(kEpi);
        tc_fence_after();
        if constexpr (MAP == FAVOR_MAP_TRIG) {
            tmem_st8(tm_addr(tmem, q, kPcAV + (NC * j) / 2), *reinterpret_cast<const uint32_t(*)[8]>(hq));
            tmem_st8(tm_addr(tmem, q, kPcAV + (NC * j + 64) / 2), *reinterpret_cast<const uint32_t(*)[8]>(hq + NC / 2));
        } else {
            tmem_st16(tm_addr(tmem, q, kPcAV + (NC * j) / 2), *reinterpret_cast<const uint32_t(*)[16]>(hq));
        }
        tmem_st_wait();
        fence_async_smem();   // KB rows (key features, state) for the tensor core
        tc_fence_before();
        mbar_arrive(e_q);
    };
    // V(c) -> fp16 with the warp's max |v| (read after the next Q, K conversion)
    auto values = [&](int c) {
        alive &= ewait(b_v, c & 1, abortp);
        float am;
        convert_tile_512<false, true>(xv, 1, e, am);
        if (am > kMaxOperand) flag_range(a.status);
        fence_async_smem();
        mbar_arrive(e_v);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        if (lane == 0) redv[(c & 1) * 16 + ew] = am;
    };
    auto take_vmax = [&](int c) {   // after a group barrier that follows values(c)
        float vm = 0.f;
#pragma unroll
        for (int i = 0; i < kEpi / 32; ++i) vm = fmaxf(vm, redv[(c & 1) * 16 + i]);
        vmax = fmaxf(vmax, vm);
    };

    // X(0) is the caller's data: convert it while the kernels before this
    // one finish; the state of the earlier segments is theirs
    if (nchunk > 0) alive &= convert_x(0);
    grid_dep_wait();
    // The states of the earlier segments come through shared memory, as in
    // tc_causal: bulk copies of the slice's 128 state rows [dv + 1] (all, or
    // 64 at a time) into the KB area, then 16 values of its row per thread.
    const uint32_t row_floats = (uint32_t)g.dv + 1;
    const int unit = (int)((uint32_t)(g.r / 64) * kKbBlk / (row_floats * 4u)) >= 128 ? 128 : 64;
    float *stg = reinterpret_cast<float *>(kb);
    int sphase = 0;
    bool staged = false;
    auto take_span = [&](const float *src, float sc) {
        for (int u = 0; u < 128; u += unit) {
            if (staged) group_sync(kEpi);   // the previous staging has been read
            if (e == 0) {
                mbar_arrive_expect_tx(bar_in, (uint32_t)unit * row_floats * 4u);
                bulk_load(stg, src + (size_t)u * row_floats, (uint32_t)unit * row_floats * 4u, bar_in);
            }
            alive &= ewait(bar_in, sphase & 1, abortp);
            ++sphase;
            staged = true;
            if (row >= u && row < u + unit) {
                const float *rp = stg + (size_t)(row - u) * row_floats;
#pragma unroll
                for (int i = 0; i < 16; ++i) s0[i] += rp[64 * dvt + 16 * j + i] * sc;
                if (j == 0) z0 += rp[g.dv] * sc;
            }
        }
    };
    if (seg > 0 && a.direct) {
        const int npin = seg * a.pps;
        const float *meta = a.meta + (size_t)bh * a.nstate * nft_full * 4 + (size_t)ft0 * 4;
        float Rs = -INFINITY;
        for (int gi = 0; gi < npin; ++gi) {
            Rs = fmaxf(Rs, meta[gi * nft_full * 4]);
            vmax = fmaxf(vmax, meta[gi * nft_full * 4 + 2]);
        }
        auto scale = [&](int gi) -> float {
            if (MAP != FAVOR_MAP_POSITIVE) return 1.f;
            const float Rg = meta[gi * nft_full * 4];
            return (Rg == -INFINITY || Rs == -INFINITY) ? 0.f : ex2(Rg - Rs);
        };
        for (int gi = 0; gi < npin; ++gi) zmax += meta[gi * nft_full * 4 + 1] * scale(gi);
        if (MAP == FAVOR_MAP_POSITIVE) R = Rs;
        const size_t per = (size_t)a.r_full * row_floats;
        for (int gi = 0; gi < npin; ++gi)
            take_span(a.state + ((size_t)bh * a.nstate + gi) * per + (size_t)ft0 * 128 * row_floats, scale(gi));
    } else if (seg > 0) {
        const float *m = a.meta_in + ((size_t)bh * a.nseg + seg) * 4;
        R = m[0];
        zmax = m[1];
        vmax = m[2];
        take_span(a.s_in + (((size_t)bh * a.nseg + seg) * a.r_full + (size_t)ft0 * 128) * row_floats, 1.f);
    }
    // the KB area is the scan's from here: every staged row has been read
    if (staged) group_sync(kEpi);
    // the ones row and the pad rows of every KB block
    for (int i = e; i < (g.r / 64) * 15 * 8; i += kEpi) {
        const int blk = i / 120, rr = kKbOne + (i % 120) / 8, ch = i % 8;
        const uint32_t one = rr == kKbOne ? 0x3C003C00u : 0u;
        *reinterpret_cast<uint4 *>(kb + (size_t)blk * kKbBlk + rr * 128 + ch * 16) = make_uint4(one, one, one, one);
    }
    fence_async_smem();
    {
        uint32_t u[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(s0[i]);
        tmem_st16(tm_addr(tmem, q, kPcS + 16 * j), u);
        if (j == 0) tmem_st1(tm_addr(tmem, q, kPcS + 64), z0);
        tmem_st_wait();
    }
    // prologue: chunk 0's key features, state rows and query features
    if (nchunk > 0) {
        const float moved = keys(0);
        if (moved != 1.f) zmax *= moved;
        state_rows(moved);
        queries(0);
        store_q();
        values(0);
        if (nchunk > 1) alive &= convert_x(1);
    }
    for (int c = 0; c < nchunk; ++c) {
        const uint32_t ph = c & 1;
        const int tc0 = t_begin + c * kC;
        const int valid = min(kC, t_end - tc0);
        const bool ok = row < valid;
        const bool more = c + 1 < nchunk;
        // ---------------- intra-chunk matrix -> masked, row-scaled, packed in place ----------------
        alive &= ewait(b_a, ph, abortp);
        tc_fence_after();
        float rho;
        {
            float av[32];
            const int limit = min(row, valid - 1) - 32 * j;   // keys j' <= limit (local index)
            float rm = 0.f;
            if (limit < 0) {
#pragma unroll
                for (int i = 0; i < 32; ++i) av[i] = 0.f;
            } else {
                tmem_ld32(tm_addr(tmem, q, kPcA + 32 * j), av);
                tmem_ld_wait();
                if (limit < 31) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) av[i] = i <= limit ? av[i] : 0.f;
                }
                float aa[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) aa[i] = fabsf(av[i]);
                rm = max_of(aa);
            }
            part2[j * 128 + row] = rm;
            group_sync(kEpi);   // also publishes the key mass of chunk c
            const float rmax = fmaxf(fmaxf(part2[row], part2[128 + row]), fmaxf(part2[256 + row], part2[384 + row]));
            rho = rmax > 0.f ? pow2_inv_floor(rmax) : 1.f;
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = pack_half2(av[2 * i] * rho, av[2 * i + 1] * rho);
            tmem_st16(tm_addr(tmem, q, kPcA + 32 * j), o);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(e_b);
        }
        {
            // chunk c's key mass and max |v| (their warp partials are complete
            // since the barrier above)
            float ms = 0.f;
#pragma unroll
            for (int i = 0; i < kEpi / 32; ++i) ms += redm[(c & 1) * 16 + i];
            zmax += ms;
            take_vmax(c);
        }
        // chunk c's scales for its output, before the next chunk moves them
        const float qoff_c = qoff_next, R_c = R, sigma_c = sigma;
        // ---------------- chunk c + 1: key features, state rows, query features ----------------
        if (more) {
            const float moved = keys(c + 1);
            if (moved != 1.f) zmax *= moved;
            state_rows(moved);
            queries(c + 1);
        }
        // ---------------- output of chunk c: the partial, sent where another CTA finalises the row ----------------
        alive &= ewait(b_av, ph, abortp);
        tc_fence_after();
        float ov[16], den, qsum = 0.f, sc = 0.f;
        bool mine = true;
        {
            float di[16], dx[16], ddi, ddx;
            tmem_ld16(tm_addr(tmem, q, kPcAV + 16 * j), di);
            tmem_ld16(tm_addr(tmem, q, kPcDX + 16 * j), dx);
            tmem_ld1(tm_addr(tmem, q, kPcAV + 64), ddi);
            tmem_ld1(tm_addr(tmem, q, kPcDD), ddx);
            if (j == 0) tmem_ld1(tm_addr(tmem, q, kPcDD + 1), qsum);
            tmem_ld_wait();
            tc_fence_before();
            const float is = pow2_inv_floor(sigma_c), ir = pow2_inv_floor(rho);   // exact: powers of two
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = fmaf(di[i], ir, dx[i] * is);
            den = fmaf(ddi, ir, ddx * is);
            if (rs > 1) {
                // each CTA's partial sits at its own scale 2^sc (query row
                // offset + key reference, log2 units); row `row` is finalised
                // by CTA row / rpo, the others send it their partial now
                sc = MAP == FAVOR_MAP_POSITIVE ? qoff_c + R_c : 0.f;
                const int owner = row / rpo;
                mine = owner == slice;
                const int slot = nslots == 2 ? (c & 1) : 0;
                if (!mine) {
                    if (nslots == 1 && c > 0) alive &= cwait(bar_free, (c - 1) & 1, abortp);
                    const int sidx = slice < owner ? slice : slice - 1, lr = row - owner * rpo;
                    const uint32_t rbar = mapa_shared(smem_u32(bar_recv(slot)), (uint32_t)owner);
                    const uint32_t rnum = mapa_shared(smem_u32(recv_num(slot, sidx, j, lr)), (uint32_t)owner);
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        st_async_v4(rnum + 16u * cc, __float_as_uint(ov[4 * cc]), __float_as_uint(ov[4 * cc + 1]),
                                    __float_as_uint(ov[4 * cc + 2]), __float_as_uint(ov[4 * cc + 3]), rbar);
                    if (j == 0)
                        st_async_v4(mapa_shared(smem_u32(recv_meta(slot, sidx, lr)), (uint32_t)owner),
                                    __float_as_uint(den), __float_as_uint(sc), __float_as_uint(qsum), 0u, rbar);
                } else if (row == slice * rpo && j == 0) {
                    mbar_arrive_expect_tx(bar_recv(slot), (uint32_t)((rs - 1) * rpo * kPartFloats * 4));
                }
            }
        }
        // ---------------- chunk c + 1: query features into TMEM; chunk c + 2: Q, K ----------------
        if (more) {
            store_q();
            if (c + 2 < nchunk) alive &= convert_x(c + 2);
        }
        // ---------------- output of chunk c: gather, normalise, store ----------------
        if (rs > 1) {
            const int slot = nslots == 2 ? (c & 1) : 0;
            if (mine) {
                alive &= cwait(bar_recv(slot), nslots == 2 ? (c >> 1) & 1 : ph, abortp);
                const int lr = row - slice * rpo;
                float smax = sc;
                for (int k2 = 0; k2 < rs - 1; ++k2) smax = fmaxf(smax, recv_meta(slot, k2, lr)[1]);
                const float wl = ex2(sc - smax);
#pragma unroll
                for (int i = 0; i < 16; ++i) ov[i] *= wl;
                den *= wl;
                qsum *= wl;
                for (int k2 = 0; k2 < rs - 1; ++k2) {
                    const float4 *pn = reinterpret_cast<const float4 *>(recv_num(slot, k2, j, lr));
                    const float4 pm = *reinterpret_cast<const float4 *>(recv_meta(slot, k2, lr));
                    const float wk = ex2(pm.y - smax);
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const float4 v4 = pn[cc];
                        ov[4 * cc] = fmaf(v4.x, wk, ov[4 * cc]);
                        ov[4 * cc + 1] = fmaf(v4.y, wk, ov[4 * cc + 1]);
                        ov[4 * cc + 2] = fmaf(v4.z, wk, ov[4 * cc + 2]);
                        ov[4 * cc + 3] = fmaf(v4.w, wk, ov[4 * cc + 3]);
                    }
                    den = fmaf(pm.x, wk, den);
                    qsum = fmaf(pm.z, wk, qsum);
                }
            }
            if (nslots == 1) {
                // the slot has been read: one arrival per owner warp at every
                // sender.  Relaxed: every value read from the slot has already
                // fed the arithmetic above, so the reads are complete when the
                // arrival is issued.
                __syncwarp();
                const int first = slice * rpo;
                if (q * 32 + 31 >= first && q * 32 < first + rpo && lane == (first & 31))
                    for (int o2 = 0; o2 < rs; ++o2)
                        if (o2 != slice) mbar_arrive_remote_relaxed(mapa_shared(smem_u32(bar_free), (uint32_t)o2));
            }
        }
        if (mine) {
            const float id = __fdividef(1.f, den);
            // the range check: the denominator against the features' fp16
            // floor (keys so far x the row sum of the query features x the
            // flush level, with a 2^10 margin)
            if (MAP == FAVOR_MAP_POSITIVE && j == 0 && ok && den < (float)(tc0 + row + 1) * qsum * kRangeFloor)
                flag_range(a.status);
            if (ok) {
                const size_t off = ((size_t)bh * a.L + tc0 + row) * g.dv + 64 * dvt + 16 * j;
                if constexpr (OB16) {
                    uint32_t h[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const __nv_bfloat162 t2 = __floats2bfloat162_rn(ov[2 * i] * id, ov[2 * i + 1] * id);
                        h[i] = *reinterpret_cast<const uint32_t *>(&t2);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + off);
                    dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
                    dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + off);
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        dst[cc] = make_float4(ov[4 * cc] * id, ov[4 * cc + 1] * id, ov[4 * cc + 2] * id, ov[4 * cc + 3] * id);
                }
            }
        }
        // ---------------- chunk c + 1: V ----------------
        if (more) values(c + 1);
    }
    if (!alive) set_status(a.status, FAVOR_ERR_TIMEOUT);
}

template <bool OB16>
__global__ void __launch_bounds__(kCausalThreads, 1)
tc_causal_split(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
                const CausalArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *small = reinterpret_cast<float *>(sm + a.o_small);
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + kSpBars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(small + kSpTslot);
    volatile int *abortp = reinterpret_cast<volatile int *>(small + kSpAbort);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        *abortp = 0;
        for (int i = 0; i < 9; ++i) mbar_init(&bars[i], 1);
        for (int i = 9; i < 15; ++i) mbar_init(&bars[i], kEpi);
        // split features: the receive slots (one local arrival + the senders'
        // bytes; slot 0 in bars[15], slot 1 in bars[17]) and the slot-free
        // barrier of a single slot (one arrival per owner warp of every
        // other CTA)
        mbar_init(&bars[15], 1);
        const int rpo = kC / a.rs;
        mbar_init(&bars[16], a.rs > 1 ? (a.rs - 1) * 4 * max(1, rpo / 32) : 1);
        mbar_init(&bars[17], 1);
        fence_mbar_init();
    }
    // ones atom after the V tile: the z column of S += phi_K^T [V | 1] and
    // the row sums of [A_m V | A_m 1]
    uint8_t *ones = sm + a.o_v + kBlk;
    for (int i = threadIdx.x; i < (int)(kBlk / 16); i += kCausalThreads)
        reinterpret_cast<uint4 *>(ones)[i] = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    if (warp == 0) tmem_alloc(tslot, a.tmem_cols);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // every CTA of a split has initialised its barriers before any remote access
    if (a.rs > 1) cluster_sync();
    const uint32_t tmem = *tslot;
    grid_dep_launch();
    if (a.g.map == FAVOR_MAP_POSITIVE) split_body<32, FAVOR_MAP_POSITIVE, OB16>(a, sm, tmem, &tm_q, &tm_k, &tm_v, &tm_out);
    else if (a.g.map == FAVOR_MAP_TRIG) split_body<16, FAVOR_MAP_TRIG, OB16>(a, sm, tmem, &tm_q, &tm_k, &tm_v, &tm_out);
    else split_body<32, FAVOR_MAP_ELU1, OB16>(a, sm, tmem, &tm_q, &tm_k, &tm_v, &tm_out);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // no CTA of a split leaves while another may still store into it
    if (a.rs > 1) cluster_sync();
    if (warp == 0) tmem_dealloc(tmem, a.tmem_cols);
}

// ---------------------------------------------------------------------------
// tc_output: non-causal rows, warp-specialised like tc_causal.  The grid is a
// flat list of (head, dv tile, 128-row chunk) units split evenly over about
// one CTA per SM; a CTA reloads W when its units move to another head and the
// state operand when they move to another (head, dv tile).  Per unit: P_Q =
// Q W^T (N = all projections) -> phi(Q) packed into TMEM -> D = phi(Q)
// [sigma KV | sigma z] (N = 64 + 16, B MN-major) -> out = D[:, :64] / D[:, 64]
// (sigma cancels).
// The units are pipelined by one: the epilogue forms the features of unit
// i + 1 in registers while the tensor core computes D(i), then writes the
// output of unit i and stores phi_Q(i + 1) into the columns D(i) has read.
// ---------------------------------------------------------------------------
struct OutputArgs {
    Geo g;
    int H, L, total_units, nq;     // nq: Q tile slots (1 or 2)
    const uint8_t *omg, *sop;      // W images; state images [BH][nvb + 1][r][64]
    int out_bf16;                  // out in bf16 (one [128][64] staging block) instead of fp32
    int *status;
    uint32_t o_w, o_s, o_x, o_stage, o_small, tmem_cols;
};

constexpr int kOutThreads = 32 + kEpi;
// the small block, in floats: row maxima [2][4][128] (by unit parity), the
// mbarriers, the TMEM slot, the abort flag
constexpr int kOutBars = 1024, kOutNumBars = 9, kOutSlot = 1044, kOutAbort = 1046, kOutSmall = 1048;
static_assert(kOutBars + 2 * kOutNumBars <= kOutSlot, "tc_output's mbarriers overlap the TMEM slot");

template <int NC, int MAP>
__device__ void output_body(const OutputArgs &a, uint8_t *sm, uint32_t tmem,
                            const CUtensorMap *tm_q, const CUtensorMap *tm_out) {
    const Geo &g = a.g;
    const int nvb = g.dv / 64, nchunk = (a.L + kC - 1) / kC;
    // units [u0, u1): an even split, CTAs differ by at most one unit
    const int u0 = (int)((long long)blockIdx.x * a.total_units / gridDim.x);
    const int u1 = (int)((long long)(blockIdx.x + 1) * a.total_units / gridDim.x);
    const int n = u1 - u0, nq = a.nq;
    const int nd = g.d / 64;
    const uint32_t xb = (uint32_t)kC * g.d * 2;
    uint8_t *w = sm + a.o_w, *sbuf = sm + a.o_s, *xs = sm + a.o_x, *stage = sm + a.o_stage;
    float *small = reinterpret_cast<float *>(sm + a.o_small);
    float *part = small;            // [2][4][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + kOutBars);
    uint64_t *bar_w = &bars[0], *bar_x = &bars[1] /*[2]*/, *bar_pq = &bars[3], *bar_d = &bars[4],
             *bar_s = &bars[5], *e_x = &bars[6], *e_p = &bars[7], *e_q = &bars[8];
    volatile int *abortp = reinterpret_cast<volatile int *>(small + kOutAbort);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // TMEM: projections [0, nproj) | D = [phi_Q sigma KV | phi_Q sigma z] [256, 336) |
    // phi_Q packed [336, 336 + r/2)
    constexpr int kColD = 256, kColPhi = 336;
    auto unit_bh = [&](int u) { return u / (nvb * nchunk); };
    auto unit_dvt = [&](int u) { return (u / nchunk) % nvb; };
    auto unit_c = [&](int u) { return u % nchunk; };
    bool alive = true;

    if (warp == 0) {
        if (lane == 0 && n == 0) grid_dep_wait();
        if (lane == 0 && n > 0) {
            const uint32_t w_s = smem_u32(w), s_s = smem_u32(sbuf), xs_s = smem_u32(xs);
            const uint32_t wbytes = (uint32_t)g.nproj * g.d * 2, atom = (uint32_t)g.r * 128;
            int wphase = 0, sphase = 0;
            auto load_w = [&](int u) {
                mbar_arrive_expect_tx(bar_w, wbytes);
                bulk_load(w, a.omg + (size_t)(unit_bh(u) % a.H) * wbytes, wbytes, bar_w);
            };
            auto load_state = [&](int u) {
                const int bh = unit_bh(u), dvt = unit_dvt(u);
                mbar_arrive_expect_tx(bar_s, 2 * atom);
                const uint8_t *img = a.sop + (size_t)bh * (nvb + 1) * atom;
                bulk_load(sbuf, img + (size_t)dvt * atom, atom, bar_s);
                bulk_load(sbuf + atom, img + (size_t)nvb * atom, atom, bar_s);
            };
            auto load_q = [&](int i) {
                const int u = u0 + i, s = i % nq;
                mbar_arrive_expect_tx(&bar_x[s], xb);
                for (int b = 0; b < nd; ++b)
                    tma_load_3d(xs + (size_t)s * xb + b * kBlk, tm_q, &bar_x[s], 64 * b, unit_c(u) * kC, unit_bh(u));
            };
            auto issue_pq = [&](int i) {
                const uint32_t x_s = xs_s + (uint32_t)(i % nq) * xb;
                const uint32_t idesc = idesc_f16(128, g.nproj, 0, 1);
                for (int kk = 0; kk < g.d / 16; ++kk)
                    mma_f16(tmem, smem_desc(x_s + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024),
                            smem_desc(w_s + kk * 2048, (uint32_t)g.d * 128, 1024), idesc, kk > 0);
                mma_commit(bar_pq);
            };
            auto key_of = [&](int u) { return unit_bh(u) * nvb + unit_dvt(u); };
            for (int i = 0; i < min(n, nq); ++i) load_q(i);
            grid_dep_wait();   // the W and state images come from the kernels before this one
            load_w(u0);
            load_state(u0);
            alive = ewait(bar_w, wphase & 1, abortp) && ewait(e_x, 0, abortp);
            ++wphase;
            if (alive) {
                tc_fence_after();
                issue_pq(0);
            }
            for (int i = 0; i < n && alive; ++i) {
                // P_Q(i) done: its Q slot takes unit i + nq
                if (!(alive = ewait(bar_pq, i & 1, abortp))) break;
                if (i + nq < n) load_q(i + nq);
                if (i + 1 < n) {
                    if (unit_bh(u0 + i + 1) != unit_bh(u0 + i)) {
                        // P_Q(i) was the last reader of the old W
                        load_w(u0 + i + 1);
                        if (!(alive = ewait(bar_w, wphase & 1, abortp))) break;
                        ++wphase;
                    }
                    // the epilogue holds P(i) in registers and has converted Q(i + 1)
                    if (!(alive = ewait(e_p, i & 1, abortp) && ewait(e_x, (i + 1) & 1, abortp))) break;
                    tc_fence_after();
                    issue_pq(i + 1);
                }
                // phi_Q(i) is in TMEM (and the epilogue has read D(i - 1))
                if (!(alive = ewait(e_q, i & 1, abortp))) break;
                if (i == 0 || key_of(u0 + i) != key_of(u0 + i - 1)) {
                    // D(i - 1) was the last reader of the old state operand
                    if (i > 0 && !(alive = ewait(bar_d, (i - 1) & 1, abortp))) break;
                    if (i > 0) load_state(u0 + i);
                    if (!(alive = ewait(bar_s, sphase & 1, abortp))) break;
                    ++sphase;
                }
                tc_fence_after();
                {
                    // D = phi_Q [sigma KV | sigma z] (B MN-major: the state atom, then the z atom)
                    const uint32_t idesc = idesc_f16(128, 80, 0, 1);
                    for (int kk = 0; kk < g.r / 16; ++kk)
                        mma_f16_ts(tmem + kColD, tmem + kColPhi + 8 * kk, smem_desc(s_s + kk * 2048, atom, 1024),
                                   idesc, kk > 0);
                    mma_commit(bar_d);
                }
            }
            if (!alive) set_status(a.status, FAVOR_ERR_TIMEOUT);
        }
        return;
    }
    const int e = threadIdx.x - 32, ew = e >> 5;
    const int q = (ew + 1) & 3, j = ew >> 2;
    const int row = q * 32 + lane;
    auto convert_x = [&](int i) -> bool {
        const bool ok = ewait(&bar_x[i % nq], (i / nq) & 1, abortp);
        float am;
        convert_tile_512<false, true>(xs + (size_t)(i % nq) * xb, nd, e, am);
        if (am > kMaxOperand) flag_range(a.status);
        tc_fence_before();
        fence_async_smem();
        mbar_arrive(e_x);
        return ok;
    };
    // the output of unit i from D(i)
    auto write_output = [&](int i) {
        const int u = u0 + i;
        alive &= ewait(bar_d, i & 1, abortp);
        tc_fence_after();
        float dn[16], dd, qs = 0.f;
        tmem_ld16(tm_addr(tmem, q, kColD + 16 * j), dn);
        tmem_ld1(tm_addr(tmem, q, kColD + 64), dd);
        if (j == 0) tmem_ld1(tm_addr(tmem, q, kColD + 65), qs);
        tmem_ld_wait();
        // the range check (sigma cancels: column 65 holds sigma x the row sum
        // of the query features)
        if (MAP == FAVOR_MAP_POSITIVE && j == 0 && unit_c(u) * kC + row < a.L &&
            dd < (float)a.L * qs * kRangeFloor)
            flag_range(a.status);
        if (e == 0) bulk_wait_read0();   // the previous unit's staging has been read
        group_sync(kEpi);
        {
            const float id = __fdividef(1.f, dd);
            if (a.out_bf16) {
                float o[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) o[i] = dn[i] * id;
                stage_bf16_16(stage, row, 16 * j, o);
            } else {
                uint8_t *halfp = stage + (size_t)((16 * j) >> 5) * kBlk;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int col = (16 * j + 4 * cc) & 31;
                    const int p = (col >> 2) ^ (row & 7);
                    *reinterpret_cast<float4 *>(halfp + row * 128 + p * 16) =
                        make_float4(dn[4 * cc] * id, dn[4 * cc + 1] * id, dn[4 * cc + 2] * id, dn[4 * cc + 3] * id);
                }
            }
        }
        fence_async_smem();
        group_sync(kEpi);
        if (e == 0 && !*abortp) {
            tma_store_3d(tm_out, stage, 64 * unit_dvt(u), unit_c(u) * kC, unit_bh(u));
            if (!a.out_bf16)
                tma_store_3d(tm_out, stage + kBlk, 64 * unit_dvt(u) + 32, unit_c(u) * kC, unit_bh(u));
            bulk_commit();
        }
    };
    if (n > 0) alive = convert_x(0);
    const uint32_t pcol = tm_addr(tmem, q, NC * j);
    // packed fp16 features of the thread's row: NC / 2 pairs (the sin/cos map:
    // NC / 2 sine pairs, then NC / 2 cosine pairs)
    constexpr int NH = MAP == FAVOR_MAP_TRIG ? NC : NC / 2;
    for (int i = 0; i < n; ++i) {
        // ---- query features of unit i -> registers ----
        alive &= ewait(bar_pq, i & 1, abortp);
        tc_fence_after();
        uint32_t hp[NH];
        if constexpr (MAP == FAVOR_MAP_POSITIVE) {
            float mx = -INFINITY;
#pragma unroll
            for (int b = 0; b < NC / 32; ++b) {
                float t32[32];
                tmem_ld32(pcol + 32 * b, t32);
                tmem_ld_wait();
                mx = fmaxf(mx, max_of(t32));
            }
            float *pm = part + (i & 1) * 512;
            pm[j * 128 + row] = mx;
            group_sync(kEpi);
            const float qoff = fmaxf(fmaxf(pm[row], pm[128 + row]), fmaxf(pm[256 + row], pm[384 + row])) - kShift;
#pragma unroll
            for (int b = 0; b < NC / 16; ++b) {
                float t16[16];
                tmem_ld16(pcol + 16 * b, t16);
                tmem_ld_wait();
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2)
                    hp[8 * b + k2] = pack_half2(ex2(t16[2 * k2] - qoff), ex2(t16[2 * k2 + 1] - qoff));
            }
        } else if constexpr (MAP == FAVOR_MAP_TRIG) {
#pragma unroll
            for (int b = 0; b < NC / 16; ++b) {
                float t16[16];
                tmem_ld16(pcol + 16 * b, t16);
                tmem_ld_wait();
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) {
                    float s0, c0, s1, c1;
                    sincos_reduced(t16[2 * k2], s0, c0);
                    sincos_reduced(t16[2 * k2 + 1], s1, c1);
                    hp[8 * b + k2] = pack_half2(s0, s1);
                    hp[NC / 2 + 8 * b + k2] = pack_half2(c0, c1);
                }
            }
        } else {
#pragma unroll
            for (int b = 0; b < NC / 16; ++b) {
                float t16[16];
                tmem_ld16(pcol + 16 * b, t16);
                tmem_ld_wait();
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) hp[8 * b + k2] = pack_half2(elu1(t16[2 * k2]), elu1(t16[2 * k2 + 1]));
            }
        }
        tc_fence_before();
        mbar_arrive(e_p);   // the projections have been read: P_Q(i + 1) may overwrite them
        // ---- next unit's Q tile (while the tensor core computes D(i - 1) and P_Q(i + 1)) ----
        if (i + 1 < n) alive &= convert_x(i + 1);
        // ---- output of unit i - 1; D(i - 1) has then read phi_Q(i - 1) ----
        if (i > 0) write_output(i - 1);
        // ---- phi_Q(i) -> TMEM [kColPhi, kColPhi + r/2) ----
        if constexpr (MAP == FAVOR_MAP_TRIG) {
            // projection p: sine at feature 128 (p / 64) + p % 64, cosine 64 further
            const int fs = 128 * ((NC * j) / 64) + (NC * j) % 64;
#pragma unroll
            for (int b = 0; b < NC / 16; ++b) {
                uint32_t os[8], oc[8];
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) {
                    os[k2] = hp[8 * b + k2];
                    oc[k2] = hp[NC / 2 + 8 * b + k2];
                }
                tmem_st8(tm_addr(tmem, q, kColPhi + (fs + 16 * b) / 2), os);
                tmem_st8(tm_addr(tmem, q, kColPhi + (fs + 64 + 16 * b) / 2), oc);
            }
        } else {
#pragma unroll
            for (int b = 0; b < NC / 16; ++b) {
                uint32_t o[8];
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) o[k2] = hp[8 * b + k2];
                tmem_st8(tm_addr(tmem, q, kColPhi + (NC * j + 16 * b) / 2), o);
            }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(e_q);
    }
    if (n > 0) write_output(n - 1);
    if (e == 0) bulk_wait0();
    if (!alive) set_status(a.status, FAVOR_ERR_TIMEOUT);
}

__global__ void __launch_bounds__(kOutThreads, 1)
tc_output(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_out,
          const OutputArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *small = reinterpret_cast<float *>(sm + a.o_small);
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + kOutBars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(small + kOutSlot);
    volatile int *abortp = reinterpret_cast<volatile int *>(small + kOutAbort);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 6; ++i) mbar_init(&bars[i], 1);
        for (int i = 6; i < kOutNumBars; ++i) mbar_init(&bars[i], kEpi);
        fence_mbar_init();
        *abortp = 0;
    }
    if (warp == 0) tmem_alloc(tslot, a.tmem_cols);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    grid_dep_launch();
    const int nc = a.g.nproj / 4;
    if (a.g.map == FAVOR_MAP_POSITIVE) {
        if (nc == 64) output_body<64, FAVOR_MAP_POSITIVE>(a, sm, tmem, &tm_q, &tm_out);
        else output_body<32, FAVOR_MAP_POSITIVE>(a, sm, tmem, &tm_q, &tm_out);
    } else if (a.g.map == FAVOR_MAP_TRIG) {
        if (nc == 32) output_body<32, FAVOR_MAP_TRIG>(a, sm, tmem, &tm_q, &tm_out);
        else output_body<16, FAVOR_MAP_TRIG>(a, sm, tmem, &tm_q, &tm_out);
    } else {
        output_body<32, FAVOR_MAP_ELU1>(a, sm, tmem, &tm_q, &tm_out);
    }
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
    uint32_t o_w, o_x, o_v, o_kb, o_small, o_recv, o_stage, bytes;
};
CausalLayout causal_layout(const Geo &g) {
    CausalLayout l;
    uint32_t o = 0;
    l.o_w = o; o = align1k(o + (uint32_t)g.nproj * g.d * 2);
    l.o_x = o; o = align1k(o + 2u * kC * g.d * 2);
    l.o_v = o; o = align1k(o + 2 * kBlk);                   // V tile + ones atom
    l.o_kb = o; o = align1k(o + (uint32_t)(g.r / 64) * kKbBlk);
    l.o_small = o; o = align1k(o + kCausalSmall * 4);
    l.o_recv = 0;
    l.o_stage = 0;
    l.bytes = o + 1024;
    return l;
}

// The pipelined scan of 128 features per CTA (tc_causal_split): g is one
// 128-feature slice; `nslots` receive slots for rs > 1
CausalLayout split_layout(const Geo &g, int rs, int nslots) {
    CausalLayout l;
    const uint32_t rpo = (uint32_t)(kC / rs);
    uint32_t o = 0;
    l.o_w = o; o = align1k(o + (uint32_t)g.nproj * g.d * 2);
    l.o_x = o; o = align1k(o + 2u * kC * g.d * 2);
    l.o_v = o; o = align1k(o + 2 * kBlk);                   // V tile + ones atom
    l.o_kb = o; o = align1k(o + 2 * kKbBlk);
    l.o_small = o; o = align1k(o + kSpSmall * 4);
    l.o_stage = 0;
    l.o_recv = o; if (rs > 1) o = align1k(o + (uint32_t)nslots * (rs - 1) * rpo * kPartFloats * 4);
    l.bytes = o + 1024;
    return l;
}

// two receive slots where they fit
int split_slots(const Geo &gs, int rs) { return split_layout(gs, rs, 2).bytes <= kSmemMax ? 2 : 1; }

// One 128-feature slice of a head: the per-CTA geometry of a split scan
// (positive and trig maps; a slice holds 128 features: 128 projections, or
// the sin and cos of 64)
Geo slice_geo(const Geo &g) {
    Geo s = g;
    s.r = 128;
    s.n_ft = 1;
    s.nproj = g.map == FAVOR_MAP_TRIG ? 64 : 128;
    return s;
}

struct StateLayout {
    uint32_t o_w, o_xk, o_xv, o_phk, o_small, xv_stride, bytes;
    int nvs, nks, FT;
};
// Feature tiles per CTA: two where TMEM holds their two state tiles beside
// the projections; then the most buffering that fits, three K and two V
// buffers first.
StateLayout state_layout(const Geo &g) {
    StateLayout l{};
    const int opts[4][2] = {{3, 2}, {2, 2}, {3, 1}, {2, 1}};
    for (int FT = (g.n_ft % 2 == 0 && 256 + 2 * (g.dv + 16) <= 512) ? 2 : 1; FT >= 1; --FT) {
        for (const auto &op : opts) {
            uint32_t o = 0;
            l.o_w = o; o = align1k(o + (uint32_t)FT * g.np_tile * g.d * 2);
            l.o_xk = o; o = align1k(o + (uint32_t)op[0] * kC * g.d * 2);
            l.xv_stride = (uint32_t)(g.dv / 64 + 1) * kBlk;       // V blocks + ones atom
            l.o_xv = o; o = align1k(o + (uint32_t)op[1] * l.xv_stride);
            l.o_phk = o; o = align1k(o + (uint32_t)FT * 2 * kBlk);
            l.o_small = o; o = align1k(o + 840 * 4);
            l.bytes = o + 1024;
            l.nks = op[0];
            l.nvs = op[1];
            l.FT = FT;
            // the final states are staged in [o_xk, o_small)
            const bool stage_fits = (size_t)FT * 128 * (g.dv + 1) * 4 <= (size_t)(l.o_small - l.o_xk);
            if (l.bytes <= kSmemMax && stage_fits) return l;
        }
    }
    return l;
}

struct OutputLayout {
    uint32_t o_w, o_s, o_x, o_stage, o_small, bytes;
    int nq;
};
OutputLayout output_layout(const Geo &g) {
    OutputLayout l;
    for (int nq = 2; nq >= 1; --nq) {
        uint32_t o = 0;
        l.o_w = o; o = align1k(o + (uint32_t)g.nproj * g.d * 2);
        l.o_s = o; o = align1k(o + 2u * g.r * 128);             // state atom + z atom
        l.o_x = o; o = align1k(o + (uint32_t)nq * kC * g.d * 2);
        l.o_stage = o; o = align1k(o + 2 * kBlk);
        l.o_small = o; o = align1k(o + kOutSmall * 4);
        l.bytes = o + 1024;
        l.nq = nq;
        if (l.bytes <= kSmemMax) break;
    }
    return l;
}

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel on the stream is still running and waits for it with
// griddepcontrol.wait before touching that kernel's results.
template <typename... KArgs, typename... Args>
int launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) != cudaSuccess) {
        cudaGetLastError();
        return FAVOR_ERR_CUDA;
    }
    return FAVOR_OK;
}

// launch_dependent with clusters of `cluster_x` CTAs along x
template <typename... KArgs, typename... Args>
int launch_dependent_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             int cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) != cudaSuccess) {
        cudaGetLastError();
        return FAVOR_ERR_CUDA;
    }
    return FAVOR_OK;
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

namespace {
// CTAs per cluster that split a head's features in the causal scan: 1 (one
// CTA holds all of them) where the whole-head layout fits, else one CTA per
// 128 features (2, 4 or 8); 0 if neither fits.
int causal_split(const Problem &p) {
    const Geo g = make_geo(p);
    if ((p.r == 128 || p.r == 256) && causal_layout(g).bytes <= kSmemMax) return 1;
    if (p.map == FAVOR_MAP_ELU1 || p.r % 128 != 0) return 0;
    const int rs = p.r / 128;
    if (rs < 2 || rs > 8) return 0;
    return split_layout(slice_geo(g), rs, 1).bytes <= kSmemMax ? rs : 0;
}

// a split head: the pipelined scan of 128 features per CTA
bool causal_pipelined(int rs) { return rs > 1; }
}  // namespace

Problem tc_widen(const Problem &p) {
    if (p.r != 64 || p.map == FAVOR_MAP_RELU || p.map == FAVOR_MAP_TRIG_SOFTMAX) return p;
    Problem w = p;
    w.omega_rows = p.nproj;
    w.nproj = 2 * p.nproj;
    w.r = 128;
    w.m = 2 * p.m;
    return w;
}

bool tc_forward_supported(const Problem &p) { return tc_supported(tc_widen(p)); }

namespace {
// the shapes the tensor-core kernels take (the host's part of tc_supported)
bool tc_shape_supported(const Problem &p) {
    // ReLU and the softmax-scaled Fourier map run on the SIMT kernels
    if (p.map == FAVOR_MAP_RELU || p.map == FAVOR_MAP_TRIG_SOFTMAX) return false;
    if (p.d != 64 && p.d != 128) return false;
    if (p.dv != 64 && p.dv != 128) return false;
    if (p.map == FAVOR_MAP_ELU1 && p.r != 128) return false;
    Geo g = make_geo(p);
    if (p.causal) {
        // wider feature sets split over the CTAs of a cluster
        if (p.r != 128 && p.r != 256 && p.r != 512 && p.r != 1024) return false;
        if (causal_split(p) == 0) return false;
    } else {
        if (p.r != 128 && p.r != 256) return false;
        if (output_layout(g).bytes > kSmemMax) return false;
    }
    return state_layout(g).bytes <= kSmemMax;
}
}  // namespace

bool tc_supported(const Problem &p) { return tc_shape_supported(p) && encoder() != nullptr; }

namespace {
struct Plan {
    int G, seg_len, nstate, pps, piece_len, nfg, nvb, nchunk;
    int rs = 1;                    // causal: CTAs per cluster splitting the features
    size_t img_bytes, per_state, bytes;
};

// Relative time of the state kernel: CTA waves x (chunks per CTA + about two
// chunks of fixed cost per CTA).
double state_cost(long ctas, int chunks, int sms) {
    return (double)((ctas + sms - 1) / sms) * (chunks + 2);
}

// The launch plan on a device of `sms` SMs (pure host arithmetic).
Plan make_plan(const Problem &p, int sms) {
    const Geo g = make_geo(p);
    Plan pl;
    pl.nvb = p.dv / 64;
    pl.nchunk = (p.L + kC - 1) / kC;
    pl.nfg = g.n_ft / state_layout(g).FT;
    if (p.causal) {
        // scan segments: whole 128-token chunks, at most one CTA per SM (a
        // split head takes rs CTAs per segment).  A scan CTA holds most of an
        // SM's shared memory, so CTAs past the SM count would run as a second
        // wave as long as the first.
        pl.rs = causal_split(p);
        const int rs = std::max(1, pl.rs);
        int G = (int)(sms / ((long long)p.BH * pl.nvb * rs));
        // at most 64 segments: the combine keeps one scale per (piece, feature tile)
        G = std::max(1, std::min(std::min(G, pl.nchunk), 64));
        const int seg_chunks = (pl.nchunk + G - 1) / G;
        pl.G = (pl.nchunk + seg_chunks - 1) / seg_chunks;
        pl.seg_len = seg_chunks * kC;
        // the states of segments 0 .. G-2 come in pieces: a divisor of the
        // segment's chunks that fills the SMs in whole waves
        int best = 1;
        double bc = 1e300;
        for (int pps = 1; pl.G > 1 && pps <= std::min(8, seg_chunks) && (pl.G - 1) * pps <= 64; ++pps) {
            if (seg_chunks % pps) continue;
            const double c = state_cost((long)p.BH * (pl.G - 1) * pps * pl.nfg, seg_chunks / pps, sms);
            if (c < bc - 1e-9) {
                bc = c;
                best = pps;
            }
        }
        pl.pps = best;
        pl.piece_len = seg_chunks / best * kC;
        pl.nstate = (pl.G - 1) * best;
    } else {
        // the state of all keys, in pieces of whole chunks that fill the SMs
        // in whole waves (the output kernel is persistent and takes no segments)
        int best = 1, best_pc = pl.nchunk;
        double bc = 1e300;
        for (int np = 1; np <= std::min(64, pl.nchunk); ++np) {
            const int pc = (pl.nchunk + np - 1) / np;
            const int npe = (pl.nchunk + pc - 1) / pc;
            const double c = state_cost((long)p.BH * npe * pl.nfg, pc, sms);
            if (c < bc - 1e-9) {
                bc = c;
                best = npe;
                best_pc = pc;
            }
        }
        pl.G = best;
        pl.seg_len = best_pc * kC;
        pl.pps = 1;
        pl.piece_len = pl.seg_len;
        pl.nstate = best;
    }
    pl.img_bytes = (size_t)p.H * p.nproj * p.d * 2;
    pl.per_state = (size_t)p.r * (p.dv + 1);
    size_t bytes = carve_bytes<uint8_t>(pl.img_bytes) +
                   carve_bytes<float>((size_t)p.BH * std::max(1, pl.nstate) * pl.per_state) +
                   carve_bytes<float>((size_t)p.BH * std::max(1, pl.nstate) * g.n_ft * 4);
    // causal: the combined segment states, only where a combine pass runs
    // (more than four segments; up to four the scan combines them itself)
    if (p.causal && pl.G > 4)
        bytes += carve_bytes<float>((size_t)p.BH * pl.G * pl.per_state) +
                 carve_bytes<float>((size_t)p.BH * pl.G * 4);
    else
        bytes += carve_bytes<uint8_t>((size_t)p.BH * (pl.nvb + 1) * p.r * 128);
    pl.bytes = bytes;
    return pl;
}

Plan make_plan(const Problem &p) { return make_plan(p, num_sms()); }

// The state pass over the plan's pieces (W image already written by
// tc_prep_omega on the same stream).
int launch_state(const Problem &p, const Geo &g, const Plan &pl, const uint8_t *img, float *state,
                 float *meta, const CUtensorMap &mk, const CUtensorMap &mv, cudaStream_t st, bool timed) {
    StateLayout sl = state_layout(g);
    StateArgs sa;
    sa.g = g; sa.H = p.H; sa.L = p.L; sa.FT = sl.FT; sa.piece_len = pl.piece_len; sa.npieces = pl.nstate;
    sa.nvs = sl.nvs; sa.nks = sl.nks;
    sa.omg = img; sa.state = state; sa.meta = meta; sa.status = device_status_ptr();
    sa.o_w = sl.o_w; sa.o_xk = sl.o_xk; sa.o_xv = sl.o_xv; sa.o_phk = sl.o_phk;
    sa.o_small = sl.o_small; sa.xv_stride = sl.xv_stride; sa.tmem_cols = 512;
    if (cudaFuncSetAttribute(tc_state, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sl.bytes) != cudaSuccess)
        return FAVOR_ERR_CUDA;
    if (timed) stats_begin(st, "tc_state");
    int rc = launch_dependent(tc_state, dim3(pl.nfg, pl.nstate, p.BH), dim3(kStateThreads), sl.bytes, st, mk, mv, sa);
    if (timed) stats_end(st);
    if (rc) return rc;
    FAVOR_LAUNCH_CHECK();
    return FAVOR_OK;
}
}  // namespace

size_t tc_scratch_bytes(const Problem &p) { return make_plan(p).bytes; }

int tc_plan_info(const Problem &p0, int sms, int *plan) {
    const Problem p = tc_widen(p0);
    if (!tc_shape_supported(p)) return FAVOR_ERR_UNSUPPORTED;
    const Plan pl = make_plan(p, sms);
    const int rs = p.causal ? std::max(1, pl.rs) : 1;
    plan[0] = pl.G;
    plan[1] = pl.pps;
    plan[2] = pl.nstate;
    plan[3] = rs;
    plan[4] = pl.nvb;
    // the scan's CTAs (causal), or the persistent output kernel's (non-causal)
    plan[5] = p.causal ? (int)std::min<long long>((long long)rs * pl.G * pl.nvb * p.BH, INT_MAX)
                       : (int)std::min<long long>((long long)pl.nchunk * p.BH * pl.nvb, sms);
    // the state pass's CTAs (0 when a causal head is one segment)
    plan[6] = (int)std::min<long long>((long long)pl.nfg * pl.nstate * p.BH, INT_MAX);
    return FAVOR_OK;
}

int tc_sincos_check(const float *x, float *s, float *c, int n, cudaStream_t st) {
    sincos_check_kernel<<<std::max(1, std::min((n + 255) / 256, 1024)), 256, 0, st>>>(x, s, c, n);
    return cuda_status(cudaGetLastError());
}

int tc_wait_expiry(long long limit_cycles, int *status, cudaStream_t st) {
    wait_expiry_kernel<<<1, 1, 0, st>>>(status, limit_cycles);
    return cuda_status(cudaGetLastError());
}

int tc_key_state(const void *k, const void *v, const float *omega, const Problem &p0, cudaStream_t st,
                 const float **state_out, const float **meta_out, int *npieces) {
    Problem p = p0;
    p.causal = 0;
    const Geo g = make_geo(p);
    const Plan pl = make_plan(p);
    int status = FAVOR_OK;
    void *ws = workspace(pl.bytes, &status);
    if (!ws) return status;
    Carve cv{static_cast<char *>(ws), 0};
    uint8_t *img = cv.take<uint8_t>(pl.img_bytes);
    float *state = cv.take<float>((size_t)p.BH * pl.nstate * pl.per_state);
    float *meta = cv.take<float>((size_t)p.BH * pl.nstate * g.n_ft * 4);
    CUtensorMap mk, mv;
    int rc;
    if ((rc = make_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.BH, p.L, p.d, 64)) ||
        (rc = make_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.BH, p.L, p.dv, 64)))
        return rc;
    tc_prep_omega<<<dim3(32, p.H), 256, 0, st>>>(omega, img, p.H, p.nproj, p.d, p.map,
                                                 p.omega_rows ? p.omega_rows : p.nproj);
    FAVOR_LAUNCH_CHECK();
    if ((rc = launch_state(p, g, pl, img, state, meta, mk, mv, st, false))) return rc;
    *state_out = state;
    *meta_out = meta;
    *npieces = pl.nstate;
    return FAVOR_OK;
}

int tc_forward(const void *q, const void *k, const void *v, const float *omega, float *out,
               const Problem &p0, cudaStream_t st) {
    const Problem p = tc_widen(p0);
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
    // the combine holds one scale per (piece, feature tile)
    if ((size_t)std::max(1, pl.nstate) * g.n_ft > (size_t)kCombineMaxTiles) return FAVOR_ERR_UNSUPPORTED;
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
    // the output box: a chunk's rows, or the rows one CTA of a split finalises
    const int out_rows = kC / (p.causal ? std::max(1, pl.rs) : 1);
    if ((rc = make_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.BH, p.L, p.d, 64)) ||
        (rc = make_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.BH, p.L, p.d, 64)) ||
        (rc = make_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.BH, p.L, p.dv, 64)) ||
        (rc = p.out_bf16 ? make_map(&mo, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.BH, p.L, p.dv, 64, out_rows)
                         : make_map(&mo, out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.BH, p.L, p.dv, 32, out_rows)))
        return rc;

    tc_prep_omega<<<dim3(32, p.H), 256, 0, st>>>(omega, img, p.H, p.nproj, p.d, p.map,
                                                 p.omega_rows ? p.omega_rows : p.nproj);
    FAVOR_LAUNCH_CHECK();

    if (nstate > 0) {
        // the state pass is the largest kernel of the non-causal path
        if ((rc = launch_state(p, g, pl, img, state, meta, mk, mv, st, !p.causal))) return rc;
    }

    if (!p.causal) {
        uint8_t *sop = cv.take<uint8_t>((size_t)p.BH * (nvb + 1) * p.r * 128);
        CombineArgs ca{};
        ca.g = g; ca.nseg = nstate; ca.pps = 1; ca.causal = 0; ca.state = state; ca.meta = meta;
        ca.sop = sop;
        ca.slice = 256;   // units of (feature, 8 value columns)
        const int nsl = (int)(((size_t)p.r * (p.dv / 8 + 1) + ca.slice - 1) / ca.slice);
        if ((rc = launch_dependent(tc_combine, dim3(p.BH, 1, nsl), dim3(256), 0, st, ca))) return rc;
        FAVOR_LAUNCH_CHECK();
        OutputLayout ol = output_layout(g);
        OutputArgs oa;
        oa.g = g; oa.H = p.H; oa.L = p.L;
        oa.total_units = nchunk * p.BH * nvb;
        oa.nq = ol.nq;
        oa.omg = img; oa.sop = sop; oa.status = dstat; oa.out_bf16 = p.out_bf16;
        oa.o_w = ol.o_w; oa.o_s = ol.o_s; oa.o_x = ol.o_x;
        oa.o_stage = ol.o_stage; oa.o_small = ol.o_small; oa.tmem_cols = 512;
        if (cudaFuncSetAttribute(tc_output, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ol.bytes) != cudaSuccess)
            return FAVOR_ERR_CUDA;
        // one persistent CTA per SM, each on a contiguous run of (head, dv tile, chunk) units
        const int grid = std::min(oa.total_units, sms);
        if ((rc = launch_dependent(tc_output, dim3(grid), dim3(kOutThreads), ol.bytes, st, mq, mo, oa))) return rc;
        FAVOR_LAUNCH_CHECK();
        return FAVOR_OK;
    }

    // up to four segments the scan kernel combines the earlier states itself
    const bool direct = G <= 4;
    float *s_in = direct ? nullptr : cv.take<float>((size_t)p.BH * G * per_state);
    float *meta_in = direct ? nullptr : cv.take<float>((size_t)p.BH * G * 4);
    if (G > 1 && !direct) {
        CombineArgs ca{};
        ca.g = g; ca.nseg = nstate; ca.pps = pl.pps; ca.causal = 1; ca.state = state; ca.meta = meta;
        ca.s_in = s_in; ca.meta_in = meta_in; ca.nout = G;
        ca.slice = 2048;
        const int nsl = (int)((per_state + ca.slice - 1) / ca.slice);
        if ((rc = launch_dependent(tc_combine, dim3(p.BH, G - 1, nsl), dim3(256), 0, st, ca))) return rc;
        FAVOR_LAUNCH_CHECK();
    }
    const int rs = std::max(1, pl.rs);
    const bool piped = causal_pipelined(rs);
    const Geo gs = piped ? slice_geo(g) : g;
    const int nslots = piped ? split_slots(gs, rs) : 1;
    CausalLayout cl = piped ? split_layout(gs, rs, nslots) : causal_layout(gs);
    CausalArgs a;
    a.g = gs;
    a.H = p.H; a.L = p.L; a.seg_len = seg_len; a.nseg = G;
    a.rs = rs; a.nft_full = g.n_ft; a.r_full = g.r;
    a.w_head_bytes = (size_t)p.nproj * p.d * 2;
    a.omg = img; a.s_in = s_in; a.meta_in = meta_in; a.status = dstat;
    a.state = state; a.meta = meta; a.nstate = nstate; a.pps = pl.pps; a.direct = direct ? 1 : 0;
    a.out_bf16 = p.out_bf16;
    a.o_w = cl.o_w; a.o_x = cl.o_x; a.o_v = cl.o_v; a.o_kb = cl.o_kb; a.o_small = cl.o_small;
    a.o_recv = cl.o_recv; a.o_stage = cl.o_stage;
    a.out = out; a.nslots = nslots;
    a.tmem_cols = 512;
    auto kern = piped ? (p.out_bf16 ? tc_causal_split<true> : tc_causal_split<false>)
                      : (p.out_bf16 ? tc_causal<true> : tc_causal<false>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cl.bytes) != cudaSuccess)
        return FAVOR_ERR_CUDA;
    stats_begin(st, piped ? "tc_causal_split" : "tc_causal");
    if ((rc = rs > 1 ? launch_dependent_cluster(kern, dim3(rs * G, nvb, p.BH), dim3(kCausalThreads), cl.bytes, st, rs,
                                                mq, mk, mv, mo, a)
                     : launch_dependent(kern, dim3(G, nvb, p.BH), dim3(kCausalThreads), cl.bytes, st, mq, mk, mv,
                                        mo, a))) {
        stats_end(st);
        return rc;
    }
    stats_end(st);
    FAVOR_LAUNCH_CHECK();
    return FAVOR_OK;
}

}  // namespace favor
