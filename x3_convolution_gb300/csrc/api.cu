// api.cu -- the extern "C" boundary of libconv3x3.so: argument validation,
// kernel-family dispatch, the device status word and driver entry points.
// The declarations, layouts and error behaviour are documented in
// include/conv3x3.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "conv3x3_internal.h"
#include "ptx.cuh"

namespace c3 {

// One status word per device, in the module's own device memory (nothing is
// allocated): kernels record CONV3X3_ERR_TIMEOUT here when a bounded wait
// gives up.
static __device__ unsigned g_status_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitNs = 2000000000ULL;  // 2 s per wait

struct DeviceInfo {
  bool ready = false;
  unsigned* status = nullptr;
  int num_sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_encodeTiled g_tiled = nullptr;
PFN_encodeIm2col g_im2col = nullptr;
bool g_entry_done = false;

void load_entry_points() {
  if (g_entry_done) return;
  g_entry_done = true;
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_tiled = reinterpret_cast<PFN_encodeTiled>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_im2col = reinterpret_cast<PFN_encodeIm2col>(fn);
}

unsigned long long wait_limit_ns() {
  static unsigned long long v = [] {
    const char* e = std::getenv("CONV3X3_WAIT_LIMIT_NS");
    unsigned long long x = e ? std::strtoull(e, nullptr, 10) : 0ULL;
    return x ? x : kDefaultWaitNs;
  }();
  return v;
}

// Device context for the current device; set-up happens on first use per device.
int get_ctx(DevCtx* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return CONV3X3_ERR_CUDA;
  if (dev >= kMaxDevices) return CONV3X3_ERR_UNSUPPORTED;  // beyond the per-device table
  std::lock_guard<std::mutex> g(g_mu);
  load_entry_points();
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return CONV3X3_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return CONV3X3_ERR_CUDA;
    di.status = static_cast<unsigned*>(p);
    di.num_sms = sms;
    di.ready = true;
  }
  out->status = di.status;
  out->num_sms = di.num_sms;
  out->wait_ns = wait_limit_ns();
  out->device = dev;
  return CONV3X3_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int check_shape(int N, int Cin, int Cout, int H, int W, bool need8) {
  if (N < 1 || H < 1 || W < 1 || Cin < 1 || Cout < 1) return CONV3X3_ERR_INVALID_ARG;
  if (need8 && (Cin % 8 != 0 || Cout % 8 != 0)) return CONV3X3_ERR_INVALID_ARG;
  if (H > 65535 || W > 65535) return CONV3X3_ERR_INVALID_ARG;
  long long P = (long long)N * H * W;
  long long C = Cin > Cout ? Cin : Cout;
  if (P * C >= (1LL << 31)) return CONV3X3_ERR_INVALID_ARG;
  return CONV3X3_OK;
}

int choose_path(int pass, const Shape& s, int path, const CatSplit& cat = CatSplit{}) {
  const bool tc = tc_supported(pass, s) && tc_supports_cat(s, cat);
  if (path == CONV3X3_PATH_SIMT) return CONV3X3_PATH_SIMT;
  if (path == CONV3X3_PATH_TENSOR) return tc ? CONV3X3_PATH_TENSOR : -1;
  return tc ? CONV3X3_PATH_TENSOR : CONV3X3_PATH_SIMT;
}

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

PFN_encodeTiled encode_tiled_fn() {
  std::lock_guard<std::mutex> g(g_mu);
  load_entry_points();
  return g_tiled;
}
PFN_encodeIm2col encode_im2col_fn() {
  std::lock_guard<std::mutex> g(g_mu);
  load_entry_points();
  return g_im2col;
}

__global__ void k_wait_selftest(unsigned* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing ever arrives on `bar`: the wait must give up and report
    mbar_wait(&bar, 0, limit_ns, status, &abort_flag);
  }
  __syncthreads();
}

bool pdl_enabled() {
  static const bool v = [] {
    const char* e = std::getenv("CONV3X3_PDL");
    return !(e && std::strcmp(e, "0") == 0);
  }();
  return v;
}

}  // namespace c3

namespace c3 {
namespace {

bool overlap(const void* a, long long abytes, const void* b, long long bbytes) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + (uintptr_t)bbytes && pb < pa + (uintptr_t)abytes;
}

// A channel split: 0 < Ca < Cin, Ca a multiple of 8, second part 16-byte aligned.
bool cat_ok(const CatSplit& cat, int Cin) {
  return !cat.on() || (cat.Ca > 0 && cat.Ca < Cin && cat.Ca % 8 == 0 && aligned16(cat.b));
}

int fwd_impl(const void* x, const void* w, const float* bias, void* y, int N, int Cin, int Cout,
             int H, int W, int act, int out_dtype, int path, const EpiExtra& ex,
             const CatSplit& cat, void* stream, int u = 1) {
  int rc = check_shape(N, Cin, Cout, H, W, true);
  if (rc) return rc;
  if (!x || !w || !y || !aligned16(x) || !aligned16(w) || !aligned16(y)) return CONV3X3_ERR_INVALID_ARG;
  if (bias && !aligned16(bias)) return CONV3X3_ERR_INVALID_ARG;
  if (act < CONV3X3_ACT_NONE || act > CONV3X3_ACT_LRELU) return CONV3X3_ERR_INVALID_ARG;
  if (out_dtype != CONV3X3_DT_BF16 && out_dtype != CONV3X3_DT_F32) return CONV3X3_ERR_INVALID_ARG;
  if (path < CONV3X3_PATH_AUTO || path > CONV3X3_PATH_SIMT) return CONV3X3_ERR_INVALID_ARG;
  if (!cat_ok(cat, Cin)) return CONV3X3_ERR_INVALID_ARG;
  if (u != 1 && u != 2) return CONV3X3_ERR_INVALID_ARG;
  Shape s{N, Cin, Cout, H, W};
  s.u = u;
  int p = choose_path(0, s, path, cat);
  if (p < 0) return CONV3X3_ERR_UNSUPPORTED;
  const int of32 = out_dtype == CONV3X3_DT_F32;
  if (p == CONV3X3_PATH_SIMT)
    return simt_fwd_bf16(x, w, bias, y, s, act, of32, ex, cat, as_stream(stream));
  DevCtx d;
  if ((rc = get_ctx(&d))) return rc;
  return tc_fwd(x, w, bias, y, s, act, of32, ex, cat, d, as_stream(stream));
}

int dgrad_impl(const void* dy, const void* w, void* dx, int N, int Cin, int Cout, int H, int W,
               int out_dtype, int path, const EpiExtra& ex, const CatSplit& cat, void* stream,
               int u = 1) {
  int rc = check_shape(N, Cin, Cout, H, W, true);
  if (rc) return rc;
  if (!dy || !w || !dx || !aligned16(dy) || !aligned16(w) || !aligned16(dx)) return CONV3X3_ERR_INVALID_ARG;
  if (out_dtype != CONV3X3_DT_BF16 && out_dtype != CONV3X3_DT_F32) return CONV3X3_ERR_INVALID_ARG;
  if (path < CONV3X3_PATH_AUTO || path > CONV3X3_PATH_SIMT) return CONV3X3_ERR_INVALID_ARG;
  if (!cat_ok(cat, Cin)) return CONV3X3_ERR_INVALID_ARG;
  if (u != 1 && u != 2) return CONV3X3_ERR_INVALID_ARG;
  Shape s{N, Cin, Cout, H, W};
  s.u = u;
  int p = choose_path(1, s, path, cat);
  if (p < 0) return CONV3X3_ERR_UNSUPPORTED;
  const int of32 = out_dtype == CONV3X3_DT_F32;
  if (p == CONV3X3_PATH_SIMT)
    return simt_dgrad_bf16(dy, w, dx, s, of32, ex, cat, as_stream(stream));
  DevCtx d;
  if ((rc = get_ctx(&d))) return rc;
  return tc_dgrad(dy, w, dx, s, of32, ex, cat, d, as_stream(stream));
}

size_t wgrad_ws_impl(int N, int Cin, int Cout, int H, int W, int path, const CatSplit& cat,
                     int u = 1) {
  if (check_shape(N, Cin, Cout, H, W, true) != CONV3X3_OK) return 0;
  if (path < CONV3X3_PATH_AUTO || path > CONV3X3_PATH_SIMT) return 0;
  if (cat.Ca != 0 && (cat.Ca < 0 || cat.Ca >= Cin || cat.Ca % 8 != 0)) return 0;
  if (u != 1 && u != 2) return 0;
  Shape s{N, Cin, Cout, H, W};
  s.u = u;
  int p = choose_path(2, s, path, cat);
  if (p < 0) return 0;
  return p == CONV3X3_PATH_SIMT ? simt_wgrad_workspace(s, 0) : tc_wgrad_workspace(s, 0);
}

int wgrad_impl(const void* x, const void* dy, float* dw, float* dbias, int N, int Cin, int Cout,
               int H, int W, void* workspace, size_t workspace_bytes, int path,
               const CatSplit& cat, void* stream, int u = 1) {
  int rc = check_shape(N, Cin, Cout, H, W, true);
  if (rc) return rc;
  if (!x || !dy || !dw || !aligned16(x) || !aligned16(dy) || !aligned16(dw)) return CONV3X3_ERR_INVALID_ARG;
  if (dbias && !aligned4(dbias)) return CONV3X3_ERR_INVALID_ARG;
  if (path < CONV3X3_PATH_AUTO || path > CONV3X3_PATH_SIMT) return CONV3X3_ERR_INVALID_ARG;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return CONV3X3_ERR_INVALID_ARG;
  if (!cat_ok(cat, Cin)) return CONV3X3_ERR_INVALID_ARG;
  if (u != 1 && u != 2) return CONV3X3_ERR_INVALID_ARG;
  Shape s{N, Cin, Cout, H, W};
  s.u = u;
  int p = choose_path(2, s, path, cat);
  if (p < 0) return CONV3X3_ERR_UNSUPPORTED;
  size_t need = p == CONV3X3_PATH_SIMT ? simt_wgrad_workspace(s, 0) : tc_wgrad_workspace(s, 0);
  if (need && (!workspace || workspace_bytes < need)) return CONV3X3_ERR_WORKSPACE;
  if (p == CONV3X3_PATH_SIMT)
    return simt_wgrad_bf16(x, dy, dw, dbias, s, workspace, workspace_bytes, 0, cat,
                           as_stream(stream));
  DevCtx d;
  if ((rc = get_ctx(&d))) return rc;
  return tc_wgrad(x, dy, dw, dbias, s, workspace, workspace_bytes, cat, d, as_stream(stream));
}

}  // namespace
}  // namespace c3

using namespace c3;

extern "C" {

const char* conv3x3_status_string(int status) {
  switch (status) {
    case CONV3X3_OK: return "ok";
    case CONV3X3_ERR_INVALID_ARG: return "invalid argument";
    case CONV3X3_ERR_UNSUPPORTED: return "unsupported by this build";
    case CONV3X3_ERR_CUDA: return "CUDA error";
    case CONV3X3_ERR_TIMEOUT: return "device wait timed out";
    case CONV3X3_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int conv3x3_auto_path(int pass, int N, int Cin, int Cout, int H, int W) {
  if (check_shape(N, Cin, Cout, H, W, true) != CONV3X3_OK) return -1;
  Shape s{N, Cin, Cout, H, W};
  return choose_path(pass, s, CONV3X3_PATH_AUTO);
}


int conv3x3_fwd_ex(const void* x, const void* w, const float* bias, void* y, int N, int Cin,
                   int Cout, int H, int W, int act, int out_dtype, int path, void* stream) {
  return fwd_impl(x, w, bias, y, N, Cin, Cout, H, W, act, out_dtype, path, EpiExtra{}, CatSplit{},
                  stream);
}

int conv3x3_fwd_save_z(const void* x, const void* w, const float* bias, void* y, void* z, int N,
                       int Cin, int Cout, int H, int W, int act, int out_dtype, int path,
                       void* stream) {
  if (!z || !aligned16(z) || !y) return CONV3X3_ERR_INVALID_ARG;
  if (check_shape(N, Cin, Cout, H, W, true) != CONV3X3_OK) return CONV3X3_ERR_INVALID_ARG;
  const long long elems = (long long)N * H * W * Cout;
  if (overlap(z, elems * 2, y, elems * (out_dtype == CONV3X3_DT_F32 ? 4 : 2)))
    return CONV3X3_ERR_INVALID_ARG;
  EpiExtra ex;
  ex.zout = z;
  return fwd_impl(x, w, bias, y, N, Cin, Cout, H, W, act, out_dtype, path, ex, CatSplit{}, stream);
}

int conv3x3_dgrad_act(const void* dy, const void* w, const void* z_in, int act_in, void* dx,
                      int N, int Cin, int Cout, int H, int W, int out_dtype, int path,
                      void* stream) {
  if (act_in < CONV3X3_ACT_NONE || act_in > CONV3X3_ACT_LRELU) return CONV3X3_ERR_INVALID_ARG;
  EpiExtra ex;
  if (act_in != CONV3X3_ACT_NONE) {
    if (!z_in || !aligned16(z_in) || !dx) return CONV3X3_ERR_INVALID_ARG;
    if (check_shape(N, Cin, Cout, H, W, true) != CONV3X3_OK) return CONV3X3_ERR_INVALID_ARG;
    const long long elems = (long long)N * H * W * Cin;
    if (overlap(z_in, elems * 2, dx, elems * (out_dtype == CONV3X3_DT_F32 ? 4 : 2)))
      return CONV3X3_ERR_INVALID_ARG;
    ex.zin = z_in;
    ex.zin_act = act_in;
  }
  return dgrad_impl(dy, w, dx, N, Cin, Cout, H, W, out_dtype, path, ex, CatSplit{}, stream);
}

int conv3x3_fwd(const void* x, const void* w, const float* bias, void* y, int N, int Cin, int Cout,
                int H, int W, int act, void* stream) {
  return conv3x3_fwd_ex(x, w, bias, y, N, Cin, Cout, H, W, act, CONV3X3_DT_BF16, CONV3X3_PATH_AUTO,
                        stream);
}

int conv3x3_dgrad_ex(const void* dy, const void* w, void* dx, int N, int Cin, int Cout, int H,
                     int W, int out_dtype, int path, void* stream) {
  return dgrad_impl(dy, w, dx, N, Cin, Cout, H, W, out_dtype, path, EpiExtra{}, CatSplit{}, stream);
}

int conv3x3_dgrad(const void* dy, const void* w, void* dx, int N, int Cin, int Cout, int H, int W,
                  void* stream) {
  return conv3x3_dgrad_ex(dy, w, dx, N, Cin, Cout, H, W, CONV3X3_DT_BF16, CONV3X3_PATH_AUTO, stream);
}

size_t conv3x3_wgrad_workspace_bytes_ex(int N, int Cin, int Cout, int H, int W, int path) {
  return wgrad_ws_impl(N, Cin, Cout, H, W, path, CatSplit{});
}

size_t conv3x3_wgrad_workspace_bytes(int N, int Cin, int Cout, int H, int W) {
  return conv3x3_wgrad_workspace_bytes_ex(N, Cin, Cout, H, W, CONV3X3_PATH_AUTO);
}

int conv3x3_wgrad_ex(const void* x, const void* dy, float* dw, float* dbias, int N, int Cin,
                     int Cout, int H, int W, void* workspace, size_t workspace_bytes, int path,
                     void* stream) {
  return wgrad_impl(x, dy, dw, dbias, N, Cin, Cout, H, W, workspace, workspace_bytes, path,
                    CatSplit{}, stream);
}

int conv3x3_fwd_cat(const void* xa, const void* xb, int Ca, const void* w, const float* bias,
                    void* y, void* z, int N, int Cin, int Cout, int H, int W, int act,
                    int out_dtype, int path, void* stream) {
  if (!xb || !y) return CONV3X3_ERR_INVALID_ARG;
  if (check_shape(N, Cin, Cout, H, W, true) != CONV3X3_OK) return CONV3X3_ERR_INVALID_ARG;
  EpiExtra ex;
  if (z) {
    if (!aligned16(z)) return CONV3X3_ERR_INVALID_ARG;
    const long long elems = (long long)N * H * W * Cout;
    if (overlap(z, elems * 2, y, elems * (out_dtype == CONV3X3_DT_F32 ? 4 : 2)))
      return CONV3X3_ERR_INVALID_ARG;
    ex.zout = z;
  }
  CatSplit cat;
  cat.b = const_cast<void*>(xb);
  cat.Ca = Ca;
  return fwd_impl(xa, w, bias, y, N, Cin, Cout, H, W, act, out_dtype, path, ex, cat, stream);
}

int conv3x3_dgrad_cat(const void* dy, const void* w, void* dxa, void* dxb, int Ca,
                      const void* za_in, const void* zb_in, int act_in, int N, int Cin, int Cout,
                      int H, int W, int out_dtype, int path, void* stream) {
  if (!dxa || !dxb) return CONV3X3_ERR_INVALID_ARG;
  if (check_shape(N, Cin, Cout, H, W, true) != CONV3X3_OK) return CONV3X3_ERR_INVALID_ARG;
  if (Ca <= 0 || Ca >= Cin || Ca % 8 != 0) return CONV3X3_ERR_INVALID_ARG;
  if (act_in < CONV3X3_ACT_NONE || act_in > CONV3X3_ACT_LRELU) return CONV3X3_ERR_INVALID_ARG;
  const long long P = (long long)N * H * W;
  const int esz = out_dtype == CONV3X3_DT_F32 ? 4 : 2;
  const long long ba = P * Ca * esz, bb = P * (Cin - Ca) * esz;
  if (overlap(dxa, ba, dxb, bb)) return CONV3X3_ERR_INVALID_ARG;
  EpiExtra ex;
  if (act_in != CONV3X3_ACT_NONE) {
    if (!za_in || !zb_in || !aligned16(za_in) || !aligned16(zb_in)) return CONV3X3_ERR_INVALID_ARG;
    const long long za = P * Ca * 2, zb = P * (Cin - Ca) * 2;
    if (overlap(za_in, za, dxa, ba) || overlap(za_in, za, dxb, bb) ||
        overlap(zb_in, zb, dxa, ba) || overlap(zb_in, zb, dxb, bb))
      return CONV3X3_ERR_INVALID_ARG;
    ex.zin = za_in;
    ex.zin_b = zb_in;
    ex.zin_act = act_in;
  }
  CatSplit cat;
  cat.b = dxb;
  cat.Ca = Ca;
  return dgrad_impl(dy, w, dxa, N, Cin, Cout, H, W, out_dtype, path, ex, cat, stream);
}

size_t conv3x3_wgrad_cat_workspace_bytes(int N, int Cin, int Ca, int Cout, int H, int W,
                                         int path) {
  if (Ca <= 0) return 0;
  CatSplit cat;
  cat.b = reinterpret_cast<void*>(uintptr_t(16));  // marks the split; never dereferenced
  cat.Ca = Ca;
  return wgrad_ws_impl(N, Cin, Cout, H, W, path, cat);
}

int conv3x3_fwd_strided(const void* x, const void* w, const float* bias, void* y, void* z, int N,
                        int Cin, int Cout, int H, int W, int stride, int act, int out_dtype,
                        int path, void* stream) {
  if (stride != 1 && stride != 2) return CONV3X3_ERR_INVALID_ARG;
  if (check_shape(N, Cin, Cout, H, W, true) != CONV3X3_OK) return CONV3X3_ERR_INVALID_ARG;
  EpiExtra ex;
  if (z) {
    if (!aligned16(z) || !y) return CONV3X3_ERR_INVALID_ARG;
    const long long elems = (long long)N * ((H - 1) / stride + 1) * ((W - 1) / stride + 1) * Cout;
    if (overlap(z, elems * 2, y, elems * (out_dtype == CONV3X3_DT_F32 ? 4 : 2)))
      return CONV3X3_ERR_INVALID_ARG;
    ex.zout = z;
  }
  return fwd_impl(x, w, bias, y, N, Cin, Cout, H, W, act, out_dtype, path, ex, CatSplit{}, stream,
                  stride);
}

int conv3x3_dgrad_strided(const void* dy, const void* w, void* dx, const void* z_in, int act_in,
                          int N, int Cin, int Cout, int H, int W, int stride, int out_dtype,
                          int path, void* stream) {
  if (stride != 1 && stride != 2) return CONV3X3_ERR_INVALID_ARG;
  if (act_in < CONV3X3_ACT_NONE || act_in > CONV3X3_ACT_LRELU) return CONV3X3_ERR_INVALID_ARG;
  EpiExtra ex;
  if (act_in != CONV3X3_ACT_NONE) {
    if (!z_in || !aligned16(z_in) || !dx) return CONV3X3_ERR_INVALID_ARG;
    if (check_shape(N, Cin, Cout, H, W, true) != CONV3X3_OK) return CONV3X3_ERR_INVALID_ARG;
    const long long elems = (long long)N * H * W * Cin;
    if (overlap(z_in, elems * 2, dx, elems * (out_dtype == CONV3X3_DT_F32 ? 4 : 2)))
      return CONV3X3_ERR_INVALID_ARG;
    ex.zin = z_in;
    ex.zin_act = act_in;
  }
  return dgrad_impl(dy, w, dx, N, Cin, Cout, H, W, out_dtype, path, ex, CatSplit{}, stream, stride);
}

size_t conv3x3_wgrad_strided_workspace_bytes(int N, int Cin, int Cout, int H, int W, int stride,
                                             int path) {
  return wgrad_ws_impl(N, Cin, Cout, H, W, path, CatSplit{}, stride);
}

int conv3x3_wgrad_strided(const void* x, const void* dy, float* dw, float* dbias, int N, int Cin,
                          int Cout, int H, int W, int stride, void* workspace,
                          size_t workspace_bytes, int path, void* stream) {
  return wgrad_impl(x, dy, dw, dbias, N, Cin, Cout, H, W, workspace, workspace_bytes, path,
                    CatSplit{}, stream, stride);
}

int conv3x3_wgrad_cat(const void* xa, const void* xb, int Ca, const void* dy, float* dw,
                      float* dbias, int N, int Cin, int Cout, int H, int W, void* workspace,
                      size_t workspace_bytes, int path, void* stream) {
  if (!xb) return CONV3X3_ERR_INVALID_ARG;
  CatSplit cat;
  cat.b = const_cast<void*>(xb);
  cat.Ca = Ca;
  return wgrad_impl(xa, dy, dw, dbias, N, Cin, Cout, H, W, workspace, workspace_bytes, path, cat,
                    stream);
}

int conv3x3_wgrad(const void* x, const void* dy, float* dw, float* dbias, int N, int Cin, int Cout,
                  int H, int W, void* workspace, size_t workspace_bytes, void* stream) {
  return conv3x3_wgrad_ex(x, dy, dw, dbias, N, Cin, Cout, H, W, workspace, workspace_bytes,
                          CONV3X3_PATH_AUTO, stream);
}

int conv3x3_fwd_f32(const float* x, const float* w, const float* bias, float* y, int N, int Cin,
                    int Cout, int H, int W, int act, void* stream) {
  int rc = check_shape(N, Cin, Cout, H, W, false);
  if (rc) return rc;
  if (!x || !w || !y || !aligned4(x) || !aligned4(w) || !aligned4(y)) return CONV3X3_ERR_INVALID_ARG;
  if (bias && !aligned4(bias)) return CONV3X3_ERR_INVALID_ARG;
  if (act < CONV3X3_ACT_NONE || act > CONV3X3_ACT_LRELU) return CONV3X3_ERR_INVALID_ARG;
  Shape s{N, Cin, Cout, H, W};
  return simt_fwd_f32(x, w, bias, y, s, act, as_stream(stream));
}

int conv3x3_dgrad_f32(const float* dy, const float* w, float* dx, int N, int Cin, int Cout, int H,
                      int W, void* stream) {
  int rc = check_shape(N, Cin, Cout, H, W, false);
  if (rc) return rc;
  if (!dy || !w || !dx || !aligned4(dy) || !aligned4(w) || !aligned4(dx)) return CONV3X3_ERR_INVALID_ARG;
  Shape s{N, Cin, Cout, H, W};
  return simt_dgrad_f32(dy, w, dx, s, as_stream(stream));
}

int conv3x3_wgrad_f32(const float* x, const float* dy, float* dw, float* dbias, int N, int Cin,
                      int Cout, int H, int W, void* workspace, size_t workspace_bytes,
                      void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  int rc = check_shape(N, Cin, Cout, H, W, false);
  if (rc) return rc;
  if (!x || !dy || !dw || !aligned4(x) || !aligned4(dy) || !aligned4(dw)) return CONV3X3_ERR_INVALID_ARG;
  if (dbias && !aligned4(dbias)) return CONV3X3_ERR_INVALID_ARG;
  Shape s{N, Cin, Cout, H, W};
  return simt_wgrad_f32(x, dy, dw, dbias, s, as_stream(stream));
}

int conv3x3_device_status(void* stream) {
  DevCtx d;
  int rc = get_ctx(&d);
  if (rc) return rc;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return CONV3X3_ERR_CUDA;
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)) != cudaSuccess) return CONV3X3_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return CONV3X3_ERR_CUDA;
  return (int)v;
}

int conv3x3_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
  DevCtx d;
  int rc = get_ctx(&d);
  if (rc) return rc;
  k_wait_selftest<<<1, 32, 0, as_stream(stream)>>>(d.status, limit_ns);
  return cudaGetLastError() == cudaSuccess ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

}  // extern "C"
