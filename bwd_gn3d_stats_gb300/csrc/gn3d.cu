// gn3d.cu -- libgn3d's C ABI: argument checks, the launch plan, per-call scratch
// and the kernel launches for GroupNorm forward and backward (see include/gn3d.h).
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>

#include <atomic>
#include <mutex>
#include <string>

#include "../../include/gn3d.h"
#include "gn3d_kernels.cuh"

namespace gn3d {
namespace {

thread_local std::string g_detail;
thread_local std::string g_msg;
std::atomic<uint64_t> g_launches{0};

int cuda_fail(cudaError_t e, const char* what) {
  g_detail = std::string(what) + ": " + cudaGetErrorString(e);
  return GN3D_ERR_CUDA;
}

int arg_fail(const char* what) {
  g_detail = what;
  return GN3D_ERR_INVALID_ARG;
}

#define GN3D_CUDA(call, what)                      \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// Per-device facts, read once.
struct DevInfo {
  bool ready = false;
  int sms = 0;
};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DevInfo g_dev[kMaxDevices];

int device_info(int dev, DevInfo* out) {
  if (dev < 0 || dev >= kMaxDevices) return arg_fail("device ordinal out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev[dev].ready) {
    GN3D_CUDA(cudaDeviceGetAttribute(&g_dev[dev].sms, cudaDevAttrMultiProcessorCount, dev),
              "cudaDeviceGetAttribute");
    g_dev[dev].ready = true;
  }
  *out = g_dev[dev];
  return GN3D_OK;
}

// A tensor argument must be device (or managed) memory of the current device.
int check_ptr(const void* p, int dev, const char* name) {
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    g_detail = std::string(name) + ": not a CUDA allocation";
    return GN3D_ERR_DEVICE;
  }
  if (a.type == cudaMemoryTypeManaged) return GN3D_OK;
  if (a.type == cudaMemoryTypeDevice && a.device == dev) return GN3D_OK;
  g_detail = std::string(name) + (a.type == cudaMemoryTypeDevice ? ": on another device"
                                                                   : ": not device memory");
  return GN3D_ERR_DEVICE;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int check_shape(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int64_t G) {
  if (N < 0 || C < 0 || D < 0 || H < 0 || W < 0) return arg_fail("negative dimension");
  if (G <= 0) return arg_fail("G must be >= 1");
  if (C % G != 0) return arg_fail("C must be divisible by G");
  // D*H*W and N*C*D*H*W must fit int64
  const double total = (double)N * (double)C * (double)D * (double)H * (double)W;
  if (total > 9.0e18) return arg_fail("tensor too large");
  if (N * (C / G) * D * H * W == 1 && C > 0)
    return arg_fail("expected more than 1 value per group (N*(C/G)*D*H*W == 1)");
  return GN3D_OK;
}

int grid_for(const DevInfo& di, int64_t units, int per_sm) {
  int64_t g = (int64_t)di.sms * per_sm;
  if (g > units) g = units;
  return (int)(g < 1 ? 1 : g);
}

template <class T>
T* carve(char*& cur, int64_t count) {
  T* p = reinterpret_cast<T*>(cur);
  cur += ((count * (int64_t)sizeof(T) + 255) / 256) * 256;
  return p;
}

// --------------------------------------------------------------- forward
template <class TI, class TO>
int launch_forward(const void* x, const float* gamma, const float* beta, const Plan& p, float eps,
                   void* y, float* mean, float* rstd, cudaStream_t st, const DevInfo& di) {
  const int64_t bytes = 256 * 4 + p.units * (int64_t)sizeof(Part) + p.NG * (int64_t)(sizeof(float4) + sizeof(unsigned));
  void* ws = nullptr;
  GN3D_CUDA(cudaMallocAsync(&ws, (size_t)bytes, st), "cudaMallocAsync(workspace)");
  char* cur = static_cast<char*>(ws);
  FwdWs w;
  w.cnt = carve<unsigned>(cur, p.NG);
  w.stats = carve<float4>(cur, p.NG);
  w.parts = carve<Part>(cur, p.units);
  cudaError_t e = cudaMemsetAsync(w.cnt, 0, (size_t)p.NG * sizeof(unsigned), st);
  if (e == cudaSuccess) {
    g_launches += 2;
    k_fwd_stats<TI><<<grid_for(di, p.units, 8), kThreads, 0, st>>>(static_cast<const TI*>(x), p, w, eps,
                                                                     mean, rstd);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    k_fwd_norm<TI, TO><<<grid_for(di, p.units, 8), kThreads, 0, st>>>(
        static_cast<const TI*>(x), static_cast<TO*>(y), p, w.stats, gamma, beta);
    e = cudaGetLastError();
  }
  cudaError_t ef = cudaFreeAsync(ws, st);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  if (ef != cudaSuccess) return cuda_fail(ef, "cudaFreeAsync(workspace)");
  return GN3D_OK;
}

// -------------------------------------------------------------- backward
template <class T>
int launch_backward(const void* dy, const void* x, const float* mean, const float* rstd,
                    const float* gamma, const Plan& p, void* dx, float* dgamma, float* dbeta,
                    cudaStream_t st, const DevInfo& di) {
  const int64_t bytes = 256 * 5 + p.units * (int64_t)sizeof(float2) + p.NC * (int64_t)sizeof(float2) +
                        p.NG * (int64_t)sizeof(float2) + (p.NG + 1) * (int64_t)sizeof(unsigned);
  void* ws = nullptr;
  GN3D_CUDA(cudaMallocAsync(&ws, (size_t)bytes, st), "cudaMallocAsync(workspace)");
  char* cur = static_cast<char*>(ws);
  BwdWs w;
  w.cnt = carve<unsigned>(cur, p.NG + 1);
  w.coef = carve<float2>(cur, p.NG);
  w.rows = carve<float2>(cur, p.NC);
  w.parts = carve<float2>(cur, p.units);
  cudaError_t e = cudaMemsetAsync(w.cnt, 0, (size_t)(p.NG + 1) * sizeof(unsigned), st);
  if (e == cudaSuccess) {
    g_launches += 2;
    k_bwd_reduce<T><<<grid_for(di, p.units, 6), kThreads, 0, st>>>(
        static_cast<const T*>(dy), static_cast<const T*>(x), p, mean, rstd, gamma, w, dgamma, dbeta);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    k_bwd_dx<T><<<grid_for(di, p.units, 6), kThreads, 0, st>>>(
        static_cast<const T*>(dy), static_cast<const T*>(x), static_cast<T*>(dx), p, mean, rstd, gamma,
        w.coef);
    e = cudaGetLastError();
  }
  cudaError_t ef = cudaFreeAsync(ws, st);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  if (ef != cudaSuccess) return cuda_fail(ef, "cudaFreeAsync(workspace)");
  return GN3D_OK;
}

bool valid_dtype(int d) { return d == GN3D_F32 || d == GN3D_BF16; }

}  // namespace
}  // namespace gn3d

using namespace gn3d;

extern "C" int gn3d_forward(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C,
                            int64_t D, int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype,
                            gn3d_dtype out_dtype, void* y, float* mean, float* rstd, void* stream) {
  int rc = check_shape(N, C, D, H, W, G);
  if (rc) return rc;
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return arg_fail("unsupported dtype");
  if (!(eps >= 0.0) || !isfinite(eps)) return arg_fail("eps must be finite and >= 0");
  const float feps = (float)eps;
  const Plan p = make_plan(N, C, D * H * W, G);
  const int64_t numel = p.NC * p.S;
  int dev = 0;
  GN3D_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  DevInfo di;
  if ((rc = device_info(dev, &di))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (numel > 0) {
    if (!x || !y) return arg_fail("x and y are required");
    if (!aligned16(x) || !aligned16(y)) return arg_fail("x and y must be 16-byte aligned");
    if ((rc = check_ptr(x, dev, "x")) || (rc = check_ptr(y, dev, "y"))) return rc;
  }
  if (p.NG > 0) {
    if (mean && (rc = check_ptr(mean, dev, "mean"))) return rc;
    if (rstd && (rc = check_ptr(rstd, dev, "rstd"))) return rc;
  }
  if (C > 0) {
    if (gamma && (rc = check_ptr(gamma, dev, "gamma"))) return rc;
    if (beta && (rc = check_ptr(beta, dev, "beta"))) return rc;
  }
  if (numel == 0) {
    if (p.NG > 0 && (mean || rstd)) {
      g_launches += 1;
      k_fill_empty_stats<<<(unsigned)((p.NG + 255) / 256), 256, 0, st>>>(mean, rstd, p.NG, feps);
      GN3D_CUDA(cudaGetLastError(), "fill launch");
    }
    return GN3D_OK;
  }
  using bf = __nv_bfloat16;
  if (in_dtype == GN3D_BF16 && out_dtype == GN3D_BF16)
    return launch_forward<bf, bf>(x, gamma, beta, p, feps, y, mean, rstd, st, di);
  if (in_dtype == GN3D_BF16 && out_dtype == GN3D_F32)
    return launch_forward<bf, float>(x, gamma, beta, p, feps, y, mean, rstd, st, di);
  if (in_dtype == GN3D_F32 && out_dtype == GN3D_BF16)
    return launch_forward<float, bf>(x, gamma, beta, p, feps, y, mean, rstd, st, di);
  return launch_forward<float, float>(x, gamma, beta, p, feps, y, mean, rstd, st, di);
}

extern "C" int gn3d_backward(const void* dy, const void* x, const float* mean, const float* rstd,
                             const float* gamma, int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                             int64_t G, gn3d_dtype dtype, void* dx, float* dgamma, float* dbeta,
                             void* stream) {
  int rc = check_shape(N, C, D, H, W, G);
  if (rc) return rc;
  if (!valid_dtype(dtype)) return arg_fail("unsupported dtype");
  const Plan p = make_plan(N, C, D * H * W, G);
  const int64_t numel = p.NC * p.S;
  int dev = 0;
  GN3D_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  DevInfo di;
  if ((rc = device_info(dev, &di))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (C > 0) {
    if (gamma && (rc = check_ptr(gamma, dev, "gamma"))) return rc;
    if (dgamma && (rc = check_ptr(dgamma, dev, "dgamma"))) return rc;
    if (dbeta && (rc = check_ptr(dbeta, dev, "dbeta"))) return rc;
  }
  if (numel == 0) {
    if (dgamma && C > 0) GN3D_CUDA(cudaMemsetAsync(dgamma, 0, (size_t)C * sizeof(float), st), "memset");
    if (dbeta && C > 0) GN3D_CUDA(cudaMemsetAsync(dbeta, 0, (size_t)C * sizeof(float), st), "memset");
    return GN3D_OK;
  }
  if (!dy || !x || !dx || !mean || !rstd) return arg_fail("dy, x, dx, mean and rstd are required");
  if (!aligned16(dy) || !aligned16(x) || !aligned16(dx)) return arg_fail("dy, x and dx must be 16-byte aligned");
  if ((rc = check_ptr(dy, dev, "dy")) || (rc = check_ptr(x, dev, "x")) || (rc = check_ptr(dx, dev, "dx")) ||
      (rc = check_ptr(mean, dev, "mean")) || (rc = check_ptr(rstd, dev, "rstd")))
    return rc;
  if (dtype == GN3D_BF16)
    return launch_backward<__nv_bfloat16>(dy, x, mean, rstd, gamma, p, dx, dgamma, dbeta, st, di);
  return launch_backward<float>(dy, x, mean, rstd, gamma, p, dx, dgamma, dbeta, st, di);
}

extern "C" int gn3d_stream_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream");
  return GN3D_OK;
}

extern "C" const char* gn3d_error_string(int status) {
  switch (status) {
    case GN3D_OK: return "ok";
    case GN3D_ERR_INVALID_ARG: g_msg = "invalid argument: " + g_detail; return g_msg.c_str();
    case GN3D_ERR_DEVICE: g_msg = "device mismatch: " + g_detail; return g_msg.c_str();
    case GN3D_ERR_CUDA: g_msg = "CUDA error: " + g_detail; return g_msg.c_str();
    case GN3D_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    default: return "unknown status";
  }
}

extern "C" uint64_t gn3d_launch_count(void) { return g_launches.load(); }

extern "C" const char* gn3d_version(void) { return "gn3d 0.1.0 sm_103a"; }
