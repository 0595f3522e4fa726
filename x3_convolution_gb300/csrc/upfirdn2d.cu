// upfirdn2d.cu -- filtered up/downsampling of NHWC bf16 activations: every
// channel is upsampled (zeros inserted after each pixel), zero-padded,
// convolved with a small FIR kernel and downsampled (every down-th pixel kept),
// the four steps of the StyleGAN2 custom-kernel blog (page titled "Dim3 grid
// calculation code", first paragraph).  Declared in include/upfirdn2d.h.
//
// No intermediate plane exists: output pixel (oy, ox) is the convolution at
// padded position (oy*down, ox*down), whose kernel taps (a, b) read the padded
// plane at (oy*down + kh-1-a, ox*down + kw-1-b).  Only positions that hold an
// input sample contribute: (oy*down + kh-1-a - pad_y0) must be a non-negative
// multiple of up inside the upsampled plane.  So the taps of row phase
// a0 = (oy*down + kh-1 - pad_y0) mod up, a0 + up, a0 + 2 up, ... are visited
// and the others skipped (polyphase): about kh/up x kw/up taps per output.
//
// The two resampling steps of a UNet (2x up and 2x down with a 4x4 filter) have
// kernels of their own in which one thread computes a 2x2 block of output
// pixels from the input samples the block shares (see below), every tap index
// known at compile time; other factors and filter sizes take the general
// kernel.
//
// The pass is bound by HBM: each thread owns 8 channels of one output pixel
// (one 16-byte load per visited tap, one 16-byte store), consecutive threads
// take consecutive channel groups and then consecutive output columns, so a
// warp reads and writes whole contiguous pixel rows; the overlap between
// neighbouring outputs' taps is served by L1/L2.  fp32 accumulation; the
// result is rounded once to bf16 on store (or written as fp32).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "conv3x3_internal.h"
#include "../../include/upfirdn2d.h"

namespace c3 {
namespace {

constexpr int kUfdThreads = 256;

struct UfdParams {
  const __nv_bfloat16* x;
  void* y;
  int N, H, W, C, Ho, Wo;
  int up, down, px0, py0, kh, kw;
  int out_f32;
  float f[UPFIRDN2D_MAX_TAPS * UPFIRDN2D_MAX_TAPS];  // [kh][kw], row pitch kw
};

__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], const uint4 v, float fv) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    acc[2 * i] = fmaf(fv, t.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(fv, t.y, acc[2 * i + 1]);
  }
}

// One output pixel's 8 channels (group cg).  UP, DOWN, KH, KW: compile-time
// factors and kernel size (0 = read them from p at run time); with all four
// fixed the tap loops unroll into predicated loads.
template <int UP, int DOWN, int KH, int KW>
__device__ __forceinline__ void ufd_point(const UfdParams& p, int n, int oy, int ox, int cg,
                                          float (&acc)[8]) {
  const int up = UP ? UP : p.up;
  const int down = DOWN ? DOWN : p.down;
  const int kh = KH ? KH : p.kh;
  const int kw = KW ? KW : p.kw;
  // padded-plane offsets of tap 0; tap (a, b) reads upsampled row ty - a,
  // column tx - b, which holds an input sample when it is a multiple of up
  const int ty = oy * down + kh - 1 - p.py0;
  const int tx = ox * down + kw - 1 - p.px0;
  int a0 = ty % up;
  if (a0 < 0) a0 += up;
  int b0 = tx % up;
  if (b0 < 0) b0 += up;
  const __nv_bfloat16* xn = p.x + (size_t)n * p.H * p.W * p.C + (size_t)cg * 8;
  // taps of one phase: a = a0, a0 + up, ... (at most ceil(kh / up) of them)
  constexpr int TA = (KH && UP) ? (KH + UP - 1) / UP : UPFIRDN2D_MAX_TAPS;
  constexpr int TB = (KW && UP) ? (KW + UP - 1) / UP : UPFIRDN2D_MAX_TAPS;
#pragma unroll
  for (int i = 0; i < TA; ++i) {
    const int a = a0 + i * up;
    if (a >= kh) break;
    const int ru = ty - a;  // decreases with a
    const int iy = ru / up;
    if (ru < 0 || iy >= p.H) continue;
    const __nv_bfloat16* xr = xn + (size_t)iy * p.W * p.C;
#pragma unroll
    for (int j = 0; j < TB; ++j) {
      const int b = b0 + j * up;
      if (b >= kw) break;
      const int cu = tx - b;
      const int ix = cu / up;
      if (cu < 0 || ix >= p.W) continue;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + (size_t)ix * p.C));
      acc_bf16x8(acc, v, p.f[a * kw + b]);
    }
  }
}

// Grid: x over 256 consecutive (output column, channel group) items of a row,
// y over bands of R output rows, z = image.  Each thread keeps its column and
// channel group and walks the R rows of its band (the index arithmetic is
// done once; the rows' loads are independent and overlap).
template <int UP, int DOWN, int KH, int KW, int R>
__global__ void __launch_bounds__(kUfdThreads)
    k_upfirdn2d(const __grid_constant__ UfdParams p) {
  // Programmatic dependent launch: the next kernel in the stream may begin
  // launching at once; nothing here reads memory before the previous kernel's
  // writes are visible.
  c3::pdl_trigger();
  c3::pdl_wait();
  const int groups = p.C >> 3;
  const int item = blockIdx.x * kUfdThreads + (int)threadIdx.x;
  if (item >= p.Wo * groups) return;
  const int ox = item / groups, cg = item - ox * groups;
  const int n = blockIdx.z;
  const int oy0 = blockIdx.y * R;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int oy = oy0 + r;
    if (oy >= p.Ho) break;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    ufd_point<UP, DOWN, KH, KW>(p, n, oy, ox, cg, acc);
    const size_t o = (((size_t)n * p.Ho + oy) * p.Wo + ox) * p.C + (size_t)cg * 8;
    if (p.out_f32) {
      float4* y4 = reinterpret_cast<float4*>(static_cast<float*>(p.y) + o);
      y4[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      y4[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      uint4 w;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) + o) = w;
    }
  }
}

// ---- 2x upsampling, 4x4 filter: polyphase 2x2 output blocks ----
// With up = 2 and kh = 4, output row oy reads upsampled rows ty - a (ty = oy +
// 3 - pad_y0) for the two taps a of its phase; when ty is even those are input
// rows ty/2 (a = 0) and ty/2 - 1 (a = 2), and row oy + 1 reads the same two
// input rows with taps 1 and 3.  So a block of output rows {oy, oy + 1} whose
// first row has ty even -- and likewise for columns -- is computed from one
// 2x2 input block:  y[oy + dy][ox + dx] = sum_{u,v} f[dy + 2u][dx + 2v] *
// x[ty/2 - u][tx/2 - v].  Four 16-byte loads serve four outputs.
// 16-byte asynchronous copy global -> shared (L1-cached); src_bytes = 0
// writes zeros without reading.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void unpack8(const uint4 v, float (&o)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void store8(const UfdParams& p, size_t o, const float (&a)[8]) {
  if (p.out_f32) {
    float4* y4 = reinterpret_cast<float4*>(static_cast<float*>(p.y) + o);
    y4[0] = make_float4(a[0], a[1], a[2], a[3]);
    y4[1] = make_float4(a[4], a[5], a[6], a[7]);
  } else {
    uint4 w;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) + o) = w;
  }
}

// Grid: x over (column block, channel group), y = row block, z = image.
__global__ void __launch_bounds__(kUfdThreads) k_upfirdn2d_up2k4(const __grid_constant__ UfdParams p) {
  c3::pdl_trigger();
  c3::pdl_wait();
  const int groups = p.C >> 3;
  const int offx = (p.px0 + 1) & 1, offy = (p.py0 + 1) & 1;  // first block starts at -1 or 0
  const int nbx = (p.Wo + offx + 1) >> 1;
  const int item = blockIdx.x * kUfdThreads + (int)threadIdx.x;
  if (item >= nbx * groups) return;
  const int bx = item / groups, cg = item - bx * groups;
  const int n = blockIdx.z;
  const int oy0 = 2 * (int)blockIdx.y - offy, ox0 = 2 * bx - offx;
  const int iy = (oy0 + 3 - p.py0) >> 1, ix = (ox0 + 3 - p.px0) >> 1;  // exact: even numerators
  const __nv_bfloat16* xn = p.x + (size_t)n * p.H * p.W * p.C + (size_t)cg * 8;
  float xv[2][2][8];
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const int r = iy - u, c = ix - v;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (r >= 0 && r < p.H && c >= 0 && c < p.W)
        w = __ldg(reinterpret_cast<const uint4*>(xn + ((size_t)r * p.W + c) * p.C));
      unpack8(w, xv[u][v]);
    }
#pragma unroll
  for (int dy = 0; dy < 2; ++dy) {
    const int oy = oy0 + dy;
    if (oy < 0 || oy >= p.Ho) continue;
#pragma unroll
    for (int dx = 0; dx < 2; ++dx) {
      const int ox = ox0 + dx;
      if (ox < 0 || ox >= p.Wo) continue;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float t = p.f[dy * 4 + dx] * xv[0][0][i];
        t = fmaf(p.f[dy * 4 + dx + 2], xv[0][1][i], t);
        t = fmaf(p.f[(dy + 2) * 4 + dx], xv[1][0][i], t);
        acc[i] = fmaf(p.f[(dy + 2) * 4 + dx + 2], xv[1][1][i], t);
      }
      store8(p, (((size_t)n * p.Ho + oy) * p.Wo + ox) * p.C + (size_t)cg * 8, acc);
    }
  }
}

// ---- 2x downsampling, 4x4 filter: 2x2 output blocks ----
// Output (oy, ox) reads input rows 2 oy + 3 - pad_y0 - a, a = 0..3 (and the
// columns likewise), so a 2x2 output block reads a 6x6 input window from row
// r0 = 2 oy0 - pad_y0: window row t serves output row dy with tap
// a = 2 dy + 3 - t when that lies in 0..3.  The window is walked row by row
// (six 16-byte loads per row), every index compile-time.
constexpr int kDownThreads = 128;
constexpr size_t kDownSmem = 36 * kDownThreads * sizeof(uint4);  // 73,728 bytes

__global__ void __launch_bounds__(kDownThreads) k_upfirdn2d_down2k4(const __grid_constant__ UfdParams p) {
  // the thread's 6x6 window, copied asynchronously into its 36 shared-memory
  // slots [slot][thread] (zeros outside the image): one memory round trip per
  // thread, where loads into registers went six rows deep in turn
  extern __shared__ uint4 win[];
  c3::pdl_trigger();
  c3::pdl_wait();
  const int groups = p.C >> 3;
  const int nbx = (p.Wo + 1) >> 1;
  const int item = blockIdx.x * kDownThreads + (int)threadIdx.x;
  if (item >= nbx * groups) return;
  const int bx = item / groups, cg = item - bx * groups;
  const int n = blockIdx.z;
  const int oy0 = 2 * (int)blockIdx.y, ox0 = 2 * bx;
  const int r0 = 2 * oy0 - p.py0, c0 = 2 * ox0 - p.px0;
  const __nv_bfloat16* xn = p.x + (size_t)n * p.H * p.W * p.C + (size_t)cg * 8;
#pragma unroll
  for (int t = 0; t < 6; ++t) {
    const int r = r0 + t;
    const bool row_ok = r >= 0 && r < p.H;
#pragma unroll
    for (int q = 0; q < 6; ++q) {
      const int c = c0 + q;
      const bool ok = row_ok && c >= 0 && c < p.W;
      cp_async16(&win[(t * 6 + q) * kDownThreads + threadIdx.x],
                 ok ? (const void*)(xn + ((size_t)r * p.W + c) * p.C) : (const void*)xn, ok ? 16 : 0);
    }
  }
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
  float acc[2][2][8];
#pragma unroll
  for (int dy = 0; dy < 2; ++dy)
#pragma unroll
    for (int dx = 0; dx < 2; ++dx)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[dy][dx][i] = 0.f;
#pragma unroll
  for (int t = 0; t < 6; ++t) {
    float xv[6][8];
#pragma unroll
    for (int q = 0; q < 6; ++q) unpack8(win[(t * 6 + q) * kDownThreads + threadIdx.x], xv[q]);
#pragma unroll
    for (int dy = 0; dy < 2; ++dy) {
      const int a = 2 * dy + 3 - t;
      if (a < 0 || a > 3) continue;  // compile-time
#pragma unroll
      for (int dx = 0; dx < 2; ++dx)
#pragma unroll
        for (int q = 0; q < 6; ++q) {
          const int b = 2 * dx + 3 - q;
          if (b < 0 || b > 3) continue;  // compile-time
          const float fv = p.f[a * 4 + b];
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[dy][dx][i] = fmaf(fv, xv[q][i], acc[dy][dx][i]);
        }
    }
  }
#pragma unroll
  for (int dy = 0; dy < 2; ++dy) {
    const int oy = oy0 + dy;
    if (oy >= p.Ho) continue;
#pragma unroll
    for (int dx = 0; dx < 2; ++dx) {
      const int ox = ox0 + dx;
      if (ox >= p.Wo) continue;
      store8(p, (((size_t)n * p.Ho + oy) * p.Wo + ox) * p.C + (size_t)cg * 8, acc[dy][dx]);
    }
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace c3

using namespace c3;

extern "C" {

int upfirdn2d_out_size(int len, int up, int down, int pad0, int pad1, int k) {
  if (len < 1 || up < 1 || up > UPFIRDN2D_MAX_FACTOR || down < 1 || down > UPFIRDN2D_MAX_FACTOR ||
      k < 1 || k > UPFIRDN2D_MAX_TAPS || pad0 < 0 || pad0 > UPFIRDN2D_MAX_PAD || pad1 < 0 ||
      pad1 > UPFIRDN2D_MAX_PAD)
    return 0;
  const long long full = (long long)len * up + pad0 + pad1 - k;
  if (full < 0) return 0;
  const long long out = full / down + 1;
  return out > 65535 ? 0 : (int)out;
}

int upfirdn2d(const void* x, const float* f, void* y, int N, int C, int H, int W, int up,
              int down, int pad_x0, int pad_x1, int pad_y0, int pad_y1, int kh, int kw,
              int out_dtype, void* stream) {
  if (N < 1 || C < 8 || C % 8 != 0 || H < 1 || W < 1 || H > 65535 || W > 65535)
    return CONV3X3_ERR_INVALID_ARG;
  const int Ho = upfirdn2d_out_size(H, up, down, pad_y0, pad_y1, kh);
  const int Wo = upfirdn2d_out_size(W, up, down, pad_x0, pad_x1, kw);
  if (Ho < 1 || Wo < 1) return CONV3X3_ERR_INVALID_ARG;
  if (!x || !y || !f || !aligned16(x) || !aligned16(y)) return CONV3X3_ERR_INVALID_ARG;
  if (out_dtype != CONV3X3_DT_BF16 && out_dtype != CONV3X3_DT_F32) return CONV3X3_ERR_INVALID_ARG;
  if ((long long)Wo * (C / 8) >= (1LL << 31)) return CONV3X3_ERR_UNSUPPORTED;  // int item index
  if (N > 65535) return CONV3X3_ERR_UNSUPPORTED;  // one grid z-slice per image
  UfdParams p;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.y = y;
  p.N = N;
  p.H = H;
  p.W = W;
  p.C = C;
  p.Ho = Ho;
  p.Wo = Wo;
  p.up = up;
  p.down = down;
  p.px0 = pad_x0;
  p.py0 = pad_y0;
  p.kh = kh;
  p.kw = kw;
  p.out_f32 = out_dtype == CONV3X3_DT_F32;
  for (int i = 0; i < kh * kw; ++i) p.f[i] = f[i];  // host taps, by value
  const long long row_items = (long long)Wo * (C / 8);
  constexpr int R = 4;  // output rows per thread
  const dim3 grid((unsigned)((row_items + kUfdThreads - 1) / kUfdThreads), (unsigned)((Ho + R - 1) / R),
                  (unsigned)N);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dim3 blk(kUfdThreads);
  cudaError_t e;
  const bool k4 = kh == 4 && kw == 4;
  const int groups = C / 8;
  if (k4 && up == 2 && down == 1) {
    const int offx = (pad_x0 + 1) & 1, offy = (pad_y0 + 1) & 1;
    const long long items = (long long)((Wo + offx + 1) / 2) * groups;
    const dim3 g2((unsigned)((items + kUfdThreads - 1) / kUfdThreads), (unsigned)((Ho + offy + 1) / 2),
                  (unsigned)N);
    e = c3::launch_pdl(k_upfirdn2d_up2k4, g2, blk, 0, st, p);
  } else if (k4 && up == 1 && down == 2) {
    const long long items = (long long)((Wo + 1) / 2) * groups;
    const dim3 g2((unsigned)((items + kDownThreads - 1) / kDownThreads), (unsigned)((Ho + 1) / 2),
                  (unsigned)N);
    // the shared-memory attribute, once per device (devices up to 64)
    static std::atomic<bool> smem_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV3X3_ERR_CUDA;
    if (dev < 0 || dev >= 64 || !smem_set[dev].load()) {
      if (cudaFuncSetAttribute(k_upfirdn2d_down2k4, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kDownSmem) != cudaSuccess)
        return CONV3X3_ERR_CUDA;
      if (dev >= 0 && dev < 64) smem_set[dev].store(true);
    }
    e = c3::launch_pdl(k_upfirdn2d_down2k4, g2, dim3(kDownThreads), kDownSmem, st, p);
  } else if (up == 1 && down == 1)
    e = c3::launch_pdl(k_upfirdn2d<1, 1, 0, 0, R>, grid, blk, 0, st, p);
  else
    e = c3::launch_pdl(k_upfirdn2d<0, 0, 0, 0, R>, grid, blk, 0, st, p);
  return e == cudaSuccess ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

}  // extern "C"
