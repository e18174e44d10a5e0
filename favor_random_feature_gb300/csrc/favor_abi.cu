// favor_abi.cu -- the extern "C" boundary of libfavor: argument validation,
// the per-device workspace, the device status word and dispatch to the
// tensor-core path (bf16 inputs) or the fp32 SIMT path.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "favor_internal.h"

namespace favor {

static __device__ int g_device_status;

namespace {

constexpr int kMaxDevices = 64;

constexpr int kHostGroups = 8;   // head groups of the host-buffer entry point
constexpr int kHostGroupsMax = kHostGroups + 2;   // the last group split twice

struct DeviceState {
    void *ws = nullptr;
    size_t ws_bytes = 0;
    void *stage = nullptr;     // host-API staging buffer
    size_t stage_bytes = 0;
    int *status = nullptr;     // device address of g_device_status
    // host-API copy streams and their events (created on first use)
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_in[kHostGroupsMax] = {}, ev_done[kHostGroupsMax] = {}, ev_out = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

int current_device(int *dev) {
    if (cudaGetDevice(dev) != cudaSuccess) return FAVOR_ERR_CUDA;
    if (*dev < 0 || *dev >= kMaxDevices) return FAVOR_ERR_UNSUPPORTED;
    return FAVOR_OK;
}

// Grow-only device buffer; frees the old one after a device sync.
void *grow(void **buf, size_t *have, size_t bytes, int *status) {
    if (*buf && *have >= bytes) return *buf;
    if (*buf) {
        cudaDeviceSynchronize();
        cudaFree(*buf);
        *buf = nullptr;
        *have = 0;
    }
    size_t want = bytes < (size_t(1) << 20) ? (size_t(1) << 20) : bytes;
    if (cudaMalloc(buf, want) != cudaSuccess) {
        cudaGetLastError();
        *buf = nullptr;
        *status = FAVOR_ERR_NOMEM;
        return nullptr;
    }
    *have = want;
    return *buf;
}

bool is_aligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t an, const void *b, size_t bn) {
    uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace

void *workspace(size_t bytes, int *status) {
    int dev;
    int rc = current_device(&dev);
    if (rc) { *status = rc; return nullptr; }
    std::lock_guard<std::mutex> lk(g_mu);
    return grow(&g_dev[dev].ws, &g_dev[dev].ws_bytes, bytes, status);
}

int *device_status_ptr() {
    int dev;
    if (current_device(&dev)) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev[dev].status) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_dev[dev].status = static_cast<int *>(p);
    }
    return g_dev[dev].status;
}

// ---- measurement hook ------------------------------------------------------
namespace {
struct Recorder {
    std::mutex mu;
    bool enabled = false;
    std::vector<cudaEvent_t> ev;   // pairs: [2i] begin, [2i+1] end
    size_t used = 0;               // events recorded so far
    const char *kernel = "";
    std::atomic<long long> launches{0};
};
Recorder g_rec;
}  // namespace

void stats_begin(cudaStream_t s, const char *kernel) {
    std::lock_guard<std::mutex> lk(g_rec.mu);
    if (!g_rec.enabled) return;
    if (g_rec.used + 2 > g_rec.ev.size()) {
        for (int i = 0; i < 2; ++i) {
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) { cudaGetLastError(); return; }
            g_rec.ev.push_back(e);
        }
    }
    g_rec.kernel = kernel;
    cudaEventRecord(g_rec.ev[g_rec.used], s);
}

void stats_end(cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_rec.mu);
    if (!g_rec.enabled || g_rec.used + 2 > g_rec.ev.size()) return;
    cudaEventRecord(g_rec.ev[g_rec.used + 1], s);
    g_rec.used += 2;
}

void stats_count_launch() {
    if (g_rec.enabled) g_rec.launches.fetch_add(1, std::memory_order_relaxed);
}

int make_problem(int B, int H, int L, int d, int dv, int m, int causal, int map, Problem *p) {
    if (B < 1 || H < 1 || L < 1) return FAVOR_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FAVOR_ERR_INVALID_ARG;
    if (map < FAVOR_MAP_POSITIVE || map > FAVOR_MAP_TRIG_SOFTMAX) return FAVOR_ERR_INVALID_ARG;
    if (d != 32 && d != 64 && d != 128) return FAVOR_ERR_UNSUPPORTED;
    if (dv != 32 && dv != 64 && dv != 128) return FAVOR_ERR_UNSUPPORTED;
    if (map_is_elementwise(map)) {
        if (m != d) return FAVOR_ERR_INVALID_ARG;
    } else {
        if (m < 1) return FAVOR_ERR_INVALID_ARG;
        if (m % 16 != 0) return FAVOR_ERR_UNSUPPORTED;
        if (m > 4096) return FAVOR_ERR_UNSUPPORTED;
    }
    long long rows = (long long)B * H * L;
    if (rows * (d > dv ? d : dv) > 0x7fffffffLL) return FAVOR_ERR_UNSUPPORTED;
    p->B = B; p->H = H; p->L = L; p->d = d; p->dv = dv; p->m = m;
    p->causal = causal;
    p->map = map;
    p->BH = B * H;
    p->nproj = map_is_elementwise(map) ? d : m;
    p->r = map_is_trig(map) ? 2 * m : (map_is_elementwise(map) ? d : m);
    return FAVOR_OK;
}

int check_ptr(const void *p, bool allow_null) {
    if (!p) return allow_null ? FAVOR_OK : FAVOR_ERR_INVALID_ARG;
    return is_aligned(p) ? FAVOR_OK : FAVOR_ERR_INVALID_ARG;
}

int validate_args(const void *q, const void *k, const void *v, const float *omega,
                  const float *out, size_t esize, const Problem &p) {
    int rc;
    if ((rc = check_ptr(q, false)) || (rc = check_ptr(k, false)) || (rc = check_ptr(v, false)) ||
        (rc = check_ptr(out, false)))
        return rc;
    if ((rc = check_ptr(omega, map_is_elementwise(p.map)))) return rc;
    size_t rows = (size_t)p.BH * p.L;
    size_t out_bytes = rows * p.dv * (p.out_bf16 ? 2 : sizeof(float));
    if (overlaps(out, out_bytes, q, rows * p.d * esize) ||
        overlaps(out, out_bytes, k, rows * p.d * esize) ||
        overlaps(out, out_bytes, v, rows * p.dv * esize) ||
        (omega && overlaps(out, out_bytes, omega, (size_t)p.H * p.nproj * p.d * sizeof(float))))
        return FAVOR_ERR_INVALID_ARG;
    return FAVOR_OK;
}

}  // namespace favor

using namespace favor;

extern "C" int favor_feature_dim(int feature_map, int d, int m) {
    if (feature_map == FAVOR_MAP_POSITIVE) return m >= 1 ? m : -1;
    if (map_is_trig(feature_map)) return m >= 1 ? 2 * m : -1;
    if (map_is_elementwise(feature_map)) return (d >= 1 && m == d) ? d : -1;
    return -1;
}

extern "C" int favor_attn_forward(const void *q, const void *k, const void *v, const float *omega,
                                  float *out, int B, int H, int L, int d, int dv, int m,
                                  int causal, int feature_map, cudaStream_t stream) {
    Problem p;
    int rc = make_problem(B, H, L, d, dv, m, causal, feature_map, &p);
    if (rc) return rc;
    if ((rc = validate_args(q, k, v, omega, out, 2, p))) return rc;
    if (tc_forward_supported(p)) return tc_forward(q, k, v, omega, out, p, stream);
    return simt_forward(q, k, v, true, omega, out, p, stream);
}

extern "C" int favor_attn_forward_bf16out(const void *q, const void *k, const void *v, const float *omega,
                                          void *out, int B, int H, int L, int d, int dv, int m, int causal,
                                          int feature_map, cudaStream_t stream) {
    Problem p;
    int rc = make_problem(B, H, L, d, dv, m, causal, feature_map, &p);
    if (rc) return rc;
    p.out_bf16 = 1;
    float *o = static_cast<float *>(out);   // bf16 storage; the kernels take the element type from p
    if ((rc = validate_args(q, k, v, omega, o, 2, p))) return rc;
    if (tc_forward_supported(p)) return tc_forward(q, k, v, omega, o, p, stream);
    return simt_forward(q, k, v, true, omega, o, p, stream);
}

extern "C" int favor_attn_forward_f32(const float *q, const float *k, const float *v,
                                      const float *omega, float *out, int B, int H, int L, int d,
                                      int dv, int m, int causal, int feature_map,
                                      cudaStream_t stream) {
    Problem p;
    int rc = make_problem(B, H, L, d, dv, m, causal, feature_map, &p);
    if (rc) return rc;
    if ((rc = validate_args(q, k, v, omega, out, 4, p))) return rc;
    return simt_forward(q, k, v, false, omega, out, p, stream);
}

namespace {
int backward_entry(const void *q, const void *k, const void *v, const float *omega, const float *dout, float *dq,
                   float *dk, float *dv, float *domega, bool bf16_in, int B, int H, int L, int d, int dv_, int m,
                   int causal, int feature_map, cudaStream_t stream) {
    Problem p;
    int rc = make_problem(B, H, L, d, dv_, m, causal, feature_map, &p);
    if (rc) return rc;
    const size_t esize = bf16_in ? 2 : 4;
    if ((rc = validate_args(q, k, v, omega, dq, esize, p))) return rc;
    if ((rc = check_ptr(dout, false)) || (rc = check_ptr(dk, false)) || (rc = check_ptr(dv, false)) ||
        (rc = check_ptr(domega, true)))
        return rc;
    const size_t rows = (size_t)p.BH * p.L;
    const void *ins[5] = {q, k, v, omega, dout};
    const size_t inb[5] = {rows * p.d * esize, rows * p.d * esize, rows * p.dv * esize,
                           omega ? (size_t)p.H * p.nproj * p.d * sizeof(float) : 0, rows * p.dv * sizeof(float)};
    const void *outs[4] = {dq, dk, dv, domega};
    const size_t outb[4] = {rows * p.d * 4, rows * p.d * 4, rows * p.dv * 4,
                            domega ? (size_t)p.H * p.nproj * p.d * sizeof(float) : 0};
    for (int i = 0; i < 4; ++i) {
        if (!outs[i]) continue;
        for (int j = 0; j < 5; ++j)
            if (ins[j] && overlaps(outs[i], outb[i], ins[j], inb[j])) return FAVOR_ERR_INVALID_ARG;
        for (int j = i + 1; j < 4; ++j)
            if (outs[j] && overlaps(outs[i], outb[i], outs[j], outb[j])) return FAVOR_ERR_INVALID_ARG;
    }
    return simt_backward(q, k, v, bf16_in, omega, dout, dq, dk, dv, domega, p, stream);
}
}  // namespace

extern "C" int favor_attn_backward(const void *q, const void *k, const void *v, const float *omega,
                                   const float *dout, float *dq, float *dk, float *dv, float *domega, int B, int H,
                                   int L, int d, int dv_, int m, int causal, int feature_map, cudaStream_t stream) {
    return backward_entry(q, k, v, omega, dout, dq, dk, dv, domega, true, B, H, L, d, dv_, m, causal, feature_map,
                          stream);
}

extern "C" int favor_attn_backward_f32(const float *q, const float *k, const float *v, const float *omega,
                                       const float *dout, float *dq, float *dk, float *dv, float *domega, int B,
                                       int H, int L, int d, int dv_, int m, int causal, int feature_map,
                                       cudaStream_t stream) {
    return backward_entry(q, k, v, omega, dout, dq, dk, dv, domega, false, B, H, L, d, dv_, m, causal, feature_map,
                          stream);
}

// The host-buffer entry point cuts the heads into up to kHostGroups groups of
// whole heads (whole batches when B allows, else head ranges of one batch) and
// pipelines them over three streams: the inputs of group g + 1 are copied in
// on s_in while group g is computed on the caller's stream and group g - 1 is
// copied out on s_out.  Each group is an independent forward pass over its
// heads (its own segment plan).
namespace {
struct HostGroup {
    int b0, nb, h0, nh;
};

int host_groups(int B, int H, HostGroup *g) {
    int n = 0;
    if (B >= kHostGroups) {
        for (int i = 0; i < kHostGroups; ++i) {
            const int b0 = (int)((long long)B * i / kHostGroups), b1 = (int)((long long)B * (i + 1) / kHostGroups);
            if (b1 > b0) g[n++] = {b0, b1 - b0, 0, H};
        }
    } else {
        const int parts = std::min(H, kHostGroups / B);
        for (int b = 0; b < B; ++b)
            for (int i = 0; i < parts; ++i) {
                const int h0 = (int)((long long)H * i / parts), h1 = (int)((long long)H * (i + 1) / parts);
                if (h1 > h0) g[n++] = {b, 1, h0, h1 - h0};
            }
    }
    // Nothing overlaps the last group's compute and copy-out: make it small.
    // Whole batches give up their last batch, and a group of one batch of
    // four or more heads its last quarter of heads.
    if (n > 0 && g[n - 1].nb > 1) {
        HostGroup &l = g[n - 1];
        g[n++] = {l.b0 + l.nb - 1, 1, 0, H};
        --l.nb;
    }
    if (n > 0 && g[n - 1].nb == 1 && g[n - 1].nh >= 4) {
        HostGroup &l = g[n - 1];
        const int q = l.nh / 4;
        g[n++] = {l.b0, 1, l.h0 + l.nh - q, q};
        l.nh -= q;
    }
    return n;
}

int host_streams(DeviceState &s) {
    if (s.s_in) return FAVOR_OK;
    bool ok = cudaStreamCreateWithFlags(&s.s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&s.s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&s.ev_out, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kHostGroupsMax; ++i)
        ok = cudaEventCreateWithFlags(&s.ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&s.ev_done[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return FAVOR_ERR_CUDA;
    }
    return FAVOR_OK;
}
}  // namespace

extern "C" int favor_attn_forward_host(const void *q, const void *k, const void *v,
                                       const float *omega, float *out, int B, int H, int L, int d,
                                       int dv, int m, int causal, int feature_map,
                                       cudaStream_t stream) {
    Problem p;
    int rc = make_problem(B, H, L, d, dv, m, causal, feature_map, &p);
    if (rc) return rc;
    if (!q || !k || !v || !out || (!omega && !map_is_elementwise(feature_map)))
        return FAVOR_ERR_INVALID_ARG;
    const size_t rows = (size_t)p.BH * p.L;
    const size_t qb = rows * p.d * 2, vb = rows * p.dv * 2, ob = rows * p.dv * 4;
    const size_t wb = omega ? (size_t)p.H * p.nproj * p.d * 4 : 0;
    const size_t need = carve_bytes<char>(qb) * 2 + carve_bytes<char>(vb) + carve_bytes<char>(wb) +
                       carve_bytes<char>(ob);
    int dev;
    if ((rc = current_device(&dev))) return rc;
    char *stage;
    DeviceState &ds = g_dev[dev];
    {
        std::lock_guard<std::mutex> lk(g_mu);
        stage = static_cast<char *>(grow(&ds.stage, &ds.stage_bytes, need, &rc));
        if (stage) rc = host_streams(ds);
    }
    if (!stage || rc) return rc ? rc : FAVOR_ERR_NOMEM;
    Carve cv{stage, 0};
    char *dq = cv.take<char>(qb), *dk = cv.take<char>(qb), *dvp = cv.take<char>(vb);
    float *dw = omega ? reinterpret_cast<float *>(cv.take<char>(wb)) : nullptr;
    float *dout = reinterpret_cast<float *>(cv.take<char>(ob));
    HostGroup grp[kHostGroupsMax];
    const int ng = host_groups(B, H, grp);
    const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k),
               *hv = static_cast<const char *>(v);
    char *hout = reinterpret_cast<char *>(out);
    // the copy streams start after the work already queued on the caller's stream
    if (cudaEventRecord(ds.ev_out, stream) != cudaSuccess || cudaStreamWaitEvent(ds.s_in, ds.ev_out, 0) != cudaSuccess ||
        cudaStreamWaitEvent(ds.s_out, ds.ev_out, 0) != cudaSuccess)
        return FAVOR_ERR_CUDA;
    if (dw && cudaMemcpyAsync(dw, omega, wb, cudaMemcpyHostToDevice, ds.s_in) != cudaSuccess) return FAVOR_ERR_CUDA;
    for (int i = 0; i < ng; ++i) {
        const HostGroup &g = grp[i];
        // rows [r0, r0 + nr) of the flattened [B H L] rows
        const size_t r0 = ((size_t)g.b0 * H + g.h0) * L, nr = (size_t)g.nb * g.nh * L;
        // whole batches: contiguous; a head range of one batch: contiguous too
        if (cudaMemcpyAsync(dq + r0 * d * 2, hq + r0 * d * 2, nr * d * 2, cudaMemcpyHostToDevice, ds.s_in) != cudaSuccess ||
            cudaMemcpyAsync(dk + r0 * d * 2, hk + r0 * d * 2, nr * d * 2, cudaMemcpyHostToDevice, ds.s_in) != cudaSuccess ||
            cudaMemcpyAsync(dvp + r0 * dv * 2, hv + r0 * dv * 2, nr * dv * 2, cudaMemcpyHostToDevice, ds.s_in) !=
                cudaSuccess ||
            cudaEventRecord(ds.ev_in[i], ds.s_in) != cudaSuccess || cudaStreamWaitEvent(stream, ds.ev_in[i], 0) != cudaSuccess)
            return FAVOR_ERR_CUDA;
        rc = favor_attn_forward(dq + r0 * d * 2, dk + r0 * d * 2, dvp + r0 * dv * 2,
                                dw ? dw + (size_t)g.h0 * p.nproj * d : nullptr, dout + r0 * dv, g.nb, g.nh, L, d, dv, m,
                                causal, feature_map, stream);
        if (rc) return rc;
        if (cudaEventRecord(ds.ev_done[i], stream) != cudaSuccess ||
            cudaStreamWaitEvent(ds.s_out, ds.ev_done[i], 0) != cudaSuccess ||
            cudaMemcpyAsync(hout + r0 * dv * 4, reinterpret_cast<char *>(dout) + r0 * dv * 4, nr * dv * 4,
                            cudaMemcpyDeviceToHost, ds.s_out) != cudaSuccess)
            return FAVOR_ERR_CUDA;
    }
    if (cudaEventRecord(ds.ev_out, ds.s_out) != cudaSuccess || cudaStreamWaitEvent(stream, ds.ev_out, 0) != cudaSuccess)
        return FAVOR_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(stream));
}

extern "C" int favor_feature_map(const void *x, const float *omega, float *phi, float *log_scale,
                                 int B, int H, int L, int d, int m, int feature_map, int is_key,
                                 cudaStream_t stream) {
    (void)is_key;
    Problem p;
    int rc = make_problem(B, H, L, d, d, m, 0, feature_map, &p);
    if (rc) return rc;
    if ((rc = check_ptr(x, false)) || (rc = check_ptr(phi, false)) ||
        (rc = check_ptr(log_scale, false)) ||
        (rc = check_ptr(omega, map_is_elementwise(feature_map))))
        return rc;
    return simt_feature_map(x, true, omega, phi, log_scale, p, stream);
}

extern "C" int favor_get_device_status(cudaStream_t stream) {
    int *sp = device_status_ptr();
    if (!sp) return FAVOR_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FAVOR_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, sp, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FAVOR_ERR_CUDA;
    int zero = 0;
    if (cudaMemcpy(sp, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FAVOR_ERR_CUDA;
    return h;
}

extern "C" int favor_plan_info(int B, int H, int L, int d, int dv, int m, int causal, int feature_map, int sms,
                               int *plan) {
    Problem p;
    int rc = make_problem(B, H, L, d, dv, m, causal, feature_map, &p);
    if (rc) return rc;
    if (!plan || sms < 1) return FAVOR_ERR_INVALID_ARG;
    return tc_plan_info(p, sms, plan);
}

extern "C" int favor_check_sincos(const float *x, float *s, float *c, int n, cudaStream_t stream) {
    if (n < 0) return FAVOR_ERR_INVALID_ARG;
    if (n == 0) return FAVOR_OK;
    int rc;
    if ((rc = check_ptr(x, false)) || (rc = check_ptr(s, false)) || (rc = check_ptr(c, false))) return rc;
    const size_t b = (size_t)n * sizeof(float);
    if (overlaps(s, b, x, b) || overlaps(c, b, x, b) || overlaps(s, b, c, b)) return FAVOR_ERR_INVALID_ARG;
    return tc_sincos_check(x, s, c, n, stream);
}

extern "C" int favor_wait_expiry_check(long long limit_cycles, cudaStream_t stream) {
    if (limit_cycles < 1 || limit_cycles > (1ll << 31)) return FAVOR_ERR_INVALID_ARG;
    int *sp = device_status_ptr();
    if (!sp) return FAVOR_ERR_CUDA;
    return tc_wait_expiry(limit_cycles, sp, stream);
}

extern "C" const char *favor_strerror(int status) {
    switch (status) {
        case FAVOR_OK: return "FAVOR_OK";
        case FAVOR_ERR_INVALID_ARG: return "FAVOR_ERR_INVALID_ARG: invalid argument";
        case FAVOR_ERR_UNSUPPORTED: return "FAVOR_ERR_UNSUPPORTED: shape not supported";
        case FAVOR_ERR_CUDA: return "FAVOR_ERR_CUDA: CUDA runtime error";
        case FAVOR_ERR_TIMEOUT: return "FAVOR_ERR_TIMEOUT: bounded device wait expired";
        case FAVOR_ERR_NOMEM: return "FAVOR_ERR_NOMEM: workspace allocation failed";
        case FAVOR_ERR_RANGE: return "FAVOR_ERR_RANGE: an input left the range of the fp16 tensor-core operands";
        default: return "unknown favor status";
    }
}

namespace favor {
namespace {
__device__ float g_ex2_sink;

// eight independent ex2 chains per thread; the feedback (y = -ex2(y)) keeps
// every operand in [-1, 0) and the chains alive
__global__ void __launch_bounds__(256) ex2_rate_kernel(int iters) {
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = -1.f - 1e-3f * (float)((threadIdx.x + i) & 63);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float y;
            asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(a[i]));
            a[i] = -y;
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += a[i];
    if (s > 0.f) g_ex2_sink = s;   // never true (s < 0): keeps the chains
}
}  // namespace
}  // namespace favor

extern "C" int favor_probe_ex2_rate(double *ex2_per_second, cudaStream_t stream) {
    if (!ex2_per_second) return FAVOR_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return FAVOR_ERR_CUDA;
    const int blocks = sms * 8, iters = 4096;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        if (e0) cudaEventDestroy(e0);
        return FAVOR_ERR_CUDA;
    }
    int rc = FAVOR_OK;
    float best = 0.f;
    for (int rep = 0; rep < 4 && rc == FAVOR_OK; ++rep) {   // the first run warms up
        cudaEventRecord(e0, stream);
        favor::ex2_rate_kernel<<<blocks, 256, 0, stream>>>(iters);
        cudaEventRecord(e1, stream);
        float ms = 0.f;
        if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
            cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
            rc = FAVOR_ERR_CUDA;
        else if (rep > 0 && (best == 0.f || ms < best))
            best = ms;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (rc) return rc;
    *ex2_per_second = (double)blocks * 256 * iters * 8 / (best * 1e-3);
    return FAVOR_OK;
}

extern "C" int favor_stats_enable(int enable) {
    std::lock_guard<std::mutex> lk(g_rec.mu);
    g_rec.enabled = enable != 0;
    if (g_rec.enabled) {
        g_rec.used = 0;
        g_rec.launches.store(0);
        g_rec.kernel = "";
    }
    return FAVOR_OK;
}

extern "C" int favor_stats_read(favor_stats_t *out) {
    if (!out) return FAVOR_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_rec.mu);
    double total = 0.0;
    for (size_t i = 0; i + 1 < g_rec.used; i += 2) {
        if (cudaEventSynchronize(g_rec.ev[i + 1]) != cudaSuccess) return FAVOR_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, g_rec.ev[i], g_rec.ev[i + 1]) != cudaSuccess)
            return FAVOR_ERR_CUDA;
        total += ms;
    }
    out->dominant_ms = total;
    out->dominant_launches = (int)(g_rec.used / 2);
    out->kernel_launches = g_rec.launches.load();
    out->dominant_kernel = g_rec.kernel;
    return FAVOR_OK;
}

extern "C" void favor_release_workspace(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (int dev = 0; dev < kMaxDevices; ++dev) {
        DeviceState &s = g_dev[dev];
        if (!s.ws && !s.stage && !s.s_in) continue;
        cudaSetDevice(dev);
        cudaDeviceSynchronize();
        if (s.ws) cudaFree(s.ws);
        if (s.stage) cudaFree(s.stage);
        s.ws = s.stage = nullptr;
        s.ws_bytes = s.stage_bytes = 0;
        if (s.s_in) {
            cudaStreamDestroy(s.s_in);
            cudaStreamDestroy(s.s_out);
            cudaEventDestroy(s.ev_out);
            for (int i = 0; i < kHostGroupsMax; ++i) {
                cudaEventDestroy(s.ev_in[i]);
                cudaEventDestroy(s.ev_done[i]);
            }
            s.s_in = s.s_out = nullptr;
            s.ev_out = nullptr;
        }
    }
    cudaSetDevice(cur);
}
