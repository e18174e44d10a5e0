// favor_internal.h -- declarations shared by the libfavor translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "favor.h"

namespace favor {

// Problem description after host validation.
struct Problem {
    int B, H, L, d, dv, m;
    int causal;
    int map;      // favor_feature_map_t
    int nproj;    // projections per token: m (positive, trig) or d (elu1)
    int r;        // feature columns: m, 2m or d
    int BH;       // B * H
    int out_bf16 = 0;   // out stored as bf16 (else fp32)
    int omega_rows = 0; // rows of the caller's omega per head (0: nproj); fewer
                        // than nproj: the projections repeat them (tc_widen)
};

// elu1, relu: r = d features straight from x (no projection); trig and its
// softmax-scaled form: 2m features, (sin, cos) per projection
__host__ __device__ inline bool map_is_elementwise(int map) { return map == FAVOR_MAP_ELU1 || map == FAVOR_MAP_RELU; }
__host__ __device__ inline bool map_is_trig(int map) { return map == FAVOR_MAP_TRIG || map == FAVOR_MAP_TRIG_SOFTMAX; }

int make_problem(int B, int H, int L, int d, int dv, int m, int causal, int map, Problem *p);
int check_ptr(const void *p, bool allow_null);

// Per-device workspace, grown on demand.  Returns nullptr on failure.
void *workspace(size_t bytes, int *status);
// Device status word (FAVOR_OK / FAVOR_ERR_TIMEOUT), written by bounded waits.
int *device_status_ptr();

// Bump allocator over a workspace block (256-byte aligned slices).
struct Carve {
    char *base;
    size_t off;
    template <typename T> T *take(size_t count) {
        size_t bytes = (count * sizeof(T) + 255) & ~size_t(255);
        T *p = reinterpret_cast<T *>(base + off);
        off += bytes;
        return p;
    }
};
template <typename T> size_t carve_bytes(size_t count) {
    return (count * sizeof(T) + 255) & ~size_t(255);
}

// SIMT path (fp32 arithmetic; input element type float or bf16 bits).
int simt_forward(const void *q, const void *k, const void *v, bool bf16_in, const float *omega,
                 float *out, const Problem &p, cudaStream_t stream);
// Backward pass on the SIMT path: g = dloss/dout [B][H][L][dv] fp32 ->
// dq, dk [B][H][L][d], dv [B][H][L][dv] and dw [H][m][d] (summed over the
// batch; skipped if null or for the elementwise maps), all fp32.
int simt_backward(const void *q, const void *k, const void *v, bool bf16_in, const float *omega, const float *g,
                  float *dq, float *dk, float *dv, float *dw, const Problem &p, cudaStream_t stream);
int simt_feature_map(const void *x, bool bf16_in, const float *omega, float *phi,
                     float *log_scale, const Problem &p, cudaStream_t stream);

// Tensor-core path (tcgen05, fp16 operands, fp32 accumulation); returns
// FAVOR_ERR_UNSUPPORTED for shapes it does not cover.
bool tc_supported(const Problem &p);
// the tensor-core epilogues' sin/cos (one range reduction + the fast sincos)
// on n device values
int tc_sincos_check(const float *x, float *s, float *c, int n, cudaStream_t st);
// A head of r = 64 features (positive m = 64, sin/cos m = 32, ELU+1 d = 64) as
// one of 128 with every projection taken twice: numerator and denominator
// both double, so the result is the same.  Other problems unchanged.
Problem tc_widen(const Problem &p);
// The forward entry points' test: the problem, widened, fits the kernels.
bool tc_forward_supported(const Problem &p);
int tc_forward(const void *q, const void *k, const void *v, const float *omega, float *out,
               const Problem &p, cudaStream_t stream);
// Scratch bytes the tensor-core path needs for a problem, and the path run on
// caller-provided scratch (FAVOR_ERR_UNSUPPORTED if ws_bytes is too small).
size_t tc_scratch_bytes(const Problem &p);
// the tensor-core launch plan of a shape on a device of `sms` SMs, without a
// device: plan[7] = segments per head (causal) or key pieces per head, pieces
// per segment, piece states per head, CTAs per head slice cluster, value
// tiles, scan or output CTAs, state CTAs.  FAVOR_ERR_UNSUPPORTED for a shape
// the tensor-core kernels do not take.
int tc_plan_info(const Problem &p, int sms, int *plan);
// One bounded mbarrier wait that nothing completes: it runs out after
// limit_cycles clock cycles and records FAVOR_ERR_TIMEOUT in *status.
int tc_wait_expiry(long long limit_cycles, int *status, cudaStream_t st);
int tc_run(const void *q, const void *k, const void *v, const float *omega, float *out,
           const Problem &p, cudaStream_t stream, void *ws, size_t ws_bytes);
// The state of all L keys of each head (non-causal state pass, no output):
// piece states [BH][npieces][r][dv+1] and their (R, max z, max|v|, max|S|)
// per 128-feature tile [BH][npieces][r/128][4], in the workspace.  Features
// are 2^(log2(e)(w.k - |k|^2/2) - R) (positive; trig sin, cos and elu1 at
// R = 0), trig features in 128-column tiles [sin 64 | cos 64].
int tc_key_state(const void *k, const void *v, const float *omega, const Problem &p, cudaStream_t st,
                 const float **state, const float **meta, int *npieces);
// The same on the SIMT path: S [BH][r][dv+1] at the per-head reference
// e^hmax[bh] (natural log), features with the 1/sqrt(m) factor, trig
// features interleaved (sin, cos) per projection.
int simt_key_state(const void *k, const void *v, bool bf16_in, const float *omega, const Problem &p,
                   cudaStream_t st, const float **S, const float **hmax);
// Host argument checks shared by the forward entry points (esize = bytes per
// q/k/v element).
int validate_args(const void *q, const void *k, const void *v, const float *omega,
                  const float *out, size_t esize, const Problem &p);

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA; }

// Measurement hook: event pair around the dominant kernel, launch counter.
void stats_begin(cudaStream_t s, const char *kernel);
void stats_end(cudaStream_t s);
void stats_count_launch();

}  // namespace favor

#define FAVOR_LAUNCH_CHECK()                                      \
    do {                                                          \
        cudaError_t e_ = cudaGetLastError();                      \
        if (e_ != cudaSuccess) return FAVOR_ERR_CUDA;             \
        ::favor::stats_count_launch();                            \
    } while (0)
