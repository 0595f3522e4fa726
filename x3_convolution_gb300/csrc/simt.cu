// simt.cu -- CUDA-core kernels for the stride-1, pad-1 3x3 convolution.
//
//  * fp32 check path (fwd / dgrad / wgrad): every tensor fp32, plain fp32 FMA,
//    one thread per output element, fixed summation order.
//  * bf16 CUDA-core path: 128-bit (8 x bf16) vector loads and stores, fp32
//    accumulation.  Cin == 8 (the UNet stem: RGB zero-padded to 8 channels) has
//    specialised kernels that keep one pixel's whole 3x3x8 window in registers
//    and the weights in shared memory; other channel counts (multiples of 8)
//    run a generic variant.  wgrad writes fixed per-split partial sums to the
//    caller's workspace and a second kernel adds them in split order, so the
//    result is bit-identical run to run.
//
// The subject page attributes its kernels' speed to vectorised loads and
// shared memory (clu0 C++/CUDA UNet diffusion, sourcepulse.org project page,
// "How It Works"); this file is that style of kernel written for sm_103a.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "act.cuh"
#include "conv3x3_internal.h"

namespace c3 {
namespace {

constexpr int kThreads = 256;
// Split plan for wgrad partial sums: a fixed constant (not the device's SM
// count) so that the workspace size and the summation order depend only on
// the shape.
constexpr int kPlanSms = 152;

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}

__device__ __forceinline__ float act_f(float z, int act) {
  if (act == CONV3X3_ACT_SILU) return z / (1.0f + __expf(-z));
  if (act == CONV3X3_ACT_LRELU) return z >= 0.0f ? z : 0.2f * z;
  return z;
}

__device__ __forceinline__ void store8(void* out, long long off, const float (&f)[8], int out_f32) {
  if (out_f32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + off);
    o[0] = make_float4(f[0], f[1], f[2], f[3]);
    o[1] = make_float4(f[4], f[5], f[6], f[7]);
  } else {
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + off) = pack8(f);
  }
}

// acc *= act'(zin[off .. off + 8)), zin bf16
__device__ __forceinline__ void scale_by_act_grad(float (&acc)[8], const __nv_bfloat16* zin,
                                                  long long off, int zin_act) {
  float z[8];
  unpack8(__ldg(reinterpret_cast<const uint4*>(zin + off)), z);
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] *= act_grad_f32(zin_act, z[i]);
}

// ======================================================================
// fp32 check path
// ======================================================================
__global__ void k_fwd_f32(const float* __restrict__ x, const float* __restrict__ w,
                          const float* __restrict__ bias, float* __restrict__ y, int N, int H,
                          int W, int Cin, int Cout, int act) {
  const long long total = (long long)N * H * W * Cout;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    int k = (int)(e % Cout);
    long long p = e / Cout;
    int ww = (int)(p % W), hh = (int)((p / W) % H), n = (int)(p / ((long long)W * H));
    float acc = bias ? bias[k] : 0.0f;
    for (int r = 0; r < 3; ++r) {
      int hi = hh + r - 1;
      if (hi < 0 || hi >= H) continue;
      for (int s = 0; s < 3; ++s) {
        int wi = ww + s - 1;
        if (wi < 0 || wi >= W) continue;
        const float* xp = x + (((long long)n * H + hi) * W + wi) * Cin;
        const float* wp = w + ((long long)(k * 3 + r) * 3 + s) * Cin;
        for (int c = 0; c < Cin; ++c) acc = __fmaf_rn(xp[c], wp[c], acc);
      }
    }
    y[e] = act_f(acc, act);
  }
}

__global__ void k_dgrad_f32(const float* __restrict__ dy, const float* __restrict__ w,
                            float* __restrict__ dx, int N, int H, int W, int Cin, int Cout) {
  const long long total = (long long)N * H * W * Cin;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    int c = (int)(e % Cin);
    long long p = e / Cin;
    int ww = (int)(p % W), hh = (int)((p / W) % H), n = (int)(p / ((long long)W * H));
    float acc = 0.0f;
    for (int r = 0; r < 3; ++r) {
      int hi = hh + 1 - r;
      if (hi < 0 || hi >= H) continue;
      for (int s = 0; s < 3; ++s) {
        int wi = ww + 1 - s;
        if (wi < 0 || wi >= W) continue;
        const float* dp = dy + (((long long)n * H + hi) * W + wi) * Cout;
        for (int k = 0; k < Cout; ++k)
          acc = __fmaf_rn(dp[k], w[((long long)(k * 3 + r) * 3 + s) * Cin + c], acc);
      }
    }
    dx[e] = acc;
  }
}

// one thread per dw element (k, r, s, c); the sum over pixels runs in order
__global__ void k_wgrad_f32(const float* __restrict__ x, const float* __restrict__ dy,
                            float* __restrict__ dw, float* __restrict__ db, int N, int H, int W,
                            int Cin, int Cout) {
  const long long total = (long long)Cout * 9 * Cin;
  const long long P = (long long)N * H * W;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    int c = (int)(e % Cin);
    int rs = (int)((e / Cin) % 9);
    int k = (int)(e / (9LL * Cin));
    int r = rs / 3, s = rs % 3;
    float acc = 0.0f;
    for (long long p = 0; p < P; ++p) {
      int ww = (int)(p % W), hh = (int)((p / W) % H);
      int hi = hh + r - 1, wi = ww + s - 1;
      if (hi < 0 || hi >= H || wi < 0 || wi >= W) continue;
      acc = __fmaf_rn(dy[p * Cout + k], x[(p + (long long)(r - 1) * W + (s - 1)) * Cin + c], acc);
    }
    dw[e] = acc;
  }
  if (db) {
    for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < Cout;
         k += (long long)gridDim.x * blockDim.x) {
      float acc = 0.0f;
      for (long long p = 0; p < P; ++p) acc += dy[p * Cout + k];
      db[k] = acc;
    }
  }
}

// ======================================================================
// bf16 CUDA-core path
// ======================================================================
// forward, Cin == 8: one thread per output pixel; the 72-value window lives in
// registers, weights (fp32, [Cout][72]) in shared memory.
__global__ void __launch_bounds__(kThreads) k_fwd_bf16_c8(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w,
    const float* __restrict__ bias, void* __restrict__ y, __nv_bfloat16* __restrict__ zout, int N,
    int H, int W, int Cout, int act, int out_f32) {
  extern __shared__ float4 smem_f4[];
  float* ws = reinterpret_cast<float*>(smem_f4);
  for (int i = threadIdx.x; i < Cout * 72; i += blockDim.x) ws[i] = __bfloat162float(w[i]);
  __syncthreads();
  const long long P = (long long)N * H * W;
  for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < P;
       p += (long long)gridDim.x * blockDim.x) {
    int ww = (int)(p % W), hh = (int)((p / W) % H);
    float in[72];
#pragma unroll
    for (int t = 0; t < 9; ++t) {
      int hi = hh + t / 3 - 1, wi = ww + t % 3 - 1;
      float f[8];
      if (hi >= 0 && hi < H && wi >= 0 && wi < W) {
        uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (p + (long long)(t / 3 - 1) * W + (t % 3 - 1)) * 8));
        unpack8(v, f);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) in[t * 8 + i] = f[i];
    }
#pragma unroll 1
    for (int k0 = 0; k0 < Cout; k0 += 8) {
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc[j] = bias ? __ldg(bias + k0 + j) : 0.0f;
        const float4* wr = reinterpret_cast<const float4*>(ws + (k0 + j) * 72);
#pragma unroll
        for (int q = 0; q < 18; ++q) {
          float4 wv = wr[q];
          acc[j] = fmaf(in[4 * q + 0], wv.x, acc[j]);
          acc[j] = fmaf(in[4 * q + 1], wv.y, acc[j]);
          acc[j] = fmaf(in[4 * q + 2], wv.z, acc[j]);
          acc[j] = fmaf(in[4 * q + 3], wv.w, acc[j]);
        }
      }
      if (zout) store8(zout, p * Cout + k0, acc, 0);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = act_f(acc[j], act);
      store8(y, p * Cout + k0, acc, out_f32);
    }
  }
}

// forward, generic Cin (multiple of 8): one thread per (pixel, 8 output channels)
// A channel-split input keeps channels [0, Ca) in x (row stride Ca) and
// [Ca, Cin) in x2 (row stride Cin - Ca); Ca = Cin when there is no split.
// Stride u: output pixel (ho, wo) of the (Ho, Wo) grid reads input pixels
// (u*ho + r - 1, u*wo + s - 1).
__global__ void __launch_bounds__(kThreads) k_fwd_bf16_gen(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ x2, int Ca,
    const __nv_bfloat16* __restrict__ w, const float* __restrict__ bias, void* __restrict__ y,
    __nv_bfloat16* __restrict__ zout, int N, int H, int W, int Cin, int Cout, int act,
    int out_f32, int u) {
  const int KG = Cout / 8;
  const int Ho = (H - 1) / u + 1, Wo = (W - 1) / u + 1;
  const long long total = (long long)N * Ho * Wo * KG;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    int k0 = (int)(e % KG) * 8;
    long long p = e / KG;
    const int wo = (int)(p % Wo), ho = (int)((p / Wo) % Ho);
    const long long n = p / ((long long)Wo * Ho);
    const int ww = u * wo, hh = u * ho;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = bias ? __ldg(bias + k0 + j) : 0.0f;
    for (int t = 0; t < 9; ++t) {
      int hi = hh + t / 3 - 1, wi = ww + t % 3 - 1;
      if (hi < 0 || hi >= H || wi < 0 || wi >= W) continue;
      const long long q = (n * H + hi) * W + wi;
      for (int c0 = 0; c0 < Cin; c0 += 8) {
        const __nv_bfloat16* xp = c0 < Ca ? x + q * Ca + c0 : x2 + q * (Cin - Ca) + (c0 - Ca);
        float xf[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(xp)), xf);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float wf[8];
          unpack8(__ldg(reinterpret_cast<const uint4*>(w + ((long long)(k0 + j) * 9 + t) * Cin + c0)), wf);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[j] = fmaf(xf[i], wf[i], acc[j]);
        }
      }
    }
    if (zout) store8(zout, p * Cout + k0, acc, 0);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = act_f(acc[j], act);
    store8(y, p * Cout + k0, acc, out_f32);
  }
}

// dgrad, Cin == 8: one thread per input pixel (8 outputs); weights as fp32
// [tap][Cout][8] in shared memory.
__global__ void __launch_bounds__(kThreads) k_dgrad_bf16_c8(
    const __nv_bfloat16* __restrict__ dy, const __nv_bfloat16* __restrict__ w,
    void* __restrict__ dx, const __nv_bfloat16* __restrict__ zin, int zin_act, int N, int H, int W,
    int Cout, int out_f32) {
  extern __shared__ float4 smem_f4[];
  float* ws = reinterpret_cast<float*>(smem_f4);
  for (int i = threadIdx.x; i < Cout * 72; i += blockDim.x) {
    int c = i % 8, t = (i / 8) % 9, k = i / 72;  // w[k][t][c]
    ws[(t * Cout + k) * 8 + c] = __bfloat162float(w[i]);
  }
  __syncthreads();
  const long long P = (long long)N * H * W;
  for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < P;
       p += (long long)gridDim.x * blockDim.x) {
    int ww = (int)(p % W), hh = (int)((p / W) % H);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll 1
    for (int t = 0; t < 9; ++t) {
      int r = t / 3, s = t % 3;
      int hi = hh + 1 - r, wi = ww + 1 - s;
      if (hi < 0 || hi >= H || wi < 0 || wi >= W) continue;
      const __nv_bfloat16* dp = dy + (p + (long long)(1 - r) * W + (1 - s)) * Cout;
      const float4* wt = reinterpret_cast<const float4*>(ws + t * Cout * 8);
#pragma unroll 1
      for (int k0 = 0; k0 < Cout; k0 += 8) {
        float d[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(dp + k0)), d);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          float4 a = wt[(k0 + kk) * 2], b = wt[(k0 + kk) * 2 + 1];
          acc[0] = fmaf(d[kk], a.x, acc[0]);
          acc[1] = fmaf(d[kk], a.y, acc[1]);
          acc[2] = fmaf(d[kk], a.z, acc[2]);
          acc[3] = fmaf(d[kk], a.w, acc[3]);
          acc[4] = fmaf(d[kk], b.x, acc[4]);
          acc[5] = fmaf(d[kk], b.y, acc[5]);
          acc[6] = fmaf(d[kk], b.z, acc[6]);
          acc[7] = fmaf(d[kk], b.w, acc[7]);
        }
      }
    }
    if (zin) scale_by_act_grad(acc, zin, p * 8, zin_act);
    store8(dx, p * 8, acc, out_f32);
  }
}

// dgrad, generic Cin: one thread per (pixel, 8 input channels)
// dx channels [0, Ca) go to dx (row stride Ca, z_in from zin), [Ca, Cin) to
// dx2 (row stride Cin - Ca, z_in from zin2); Ca = Cin when there is no split.
__global__ void __launch_bounds__(kThreads) k_dgrad_bf16_gen(
    const __nv_bfloat16* __restrict__ dy, const __nv_bfloat16* __restrict__ w,
    void* __restrict__ dx, void* __restrict__ dx2, int Ca, const __nv_bfloat16* __restrict__ zin,
    const __nv_bfloat16* __restrict__ zin2, int zin_act, int N, int H, int W, int Cin, int Cout,
    int out_f32, int u) {
  const int CG = Cin / 8;
  const int Ho = (H - 1) / u + 1, Wo = (W - 1) / u + 1;
  const long long total = (long long)N * H * W * CG;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    int c0 = (int)(e % CG) * 8;
    long long p = e / CG;
    int ww = (int)(p % W), hh = (int)((p / W) % H);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    const long long n = p / ((long long)W * H);
    for (int t = 0; t < 9; ++t) {
      int r = t / 3, s = t % 3;
      // dy pixel (ho, wo) with u*ho + r - 1 = hh and u*wo + s - 1 = ww
      int th = hh + 1 - r, tw = ww + 1 - s;
      if (th < 0 || tw < 0 || th % u != 0 || tw % u != 0) continue;
      int hi = th / u, wi = tw / u;
      if (hi >= Ho || wi >= Wo) continue;
      const __nv_bfloat16* dp = dy + ((n * Ho + hi) * Wo + wi) * Cout;
      for (int k0 = 0; k0 < Cout; k0 += 8) {
        float d[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(dp + k0)), d);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          float wf[8];
          unpack8(__ldg(reinterpret_cast<const uint4*>(w + ((long long)(k0 + kk) * 9 + t) * Cin + c0)), wf);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(d[kk], wf[i], acc[i]);
        }
      }
    }
    const bool second = c0 >= Ca;
    const long long off = second ? p * (Cin - Ca) + (c0 - Ca) : p * Ca + c0;
    if (zin) scale_by_act_grad(acc, second ? zin2 : zin, off, zin_act);
    store8(second ? dx2 : dx, off, acc, out_f32);
  }
}

// wgrad partial sums.  Split `s` (blockIdx.y) owns pixels [s*chunk, (s+1)*chunk).
// One thread per (k, tap, 8 input channels): its 8 running sums cover
// dw[k][tap][c0..c0+8).  Threads with a block-wide index below Cout also sum
// dbias.  partial layout: [S][Cout*9*Cin] followed by [S][Cout].
__global__ void __launch_bounds__(kThreads) k_wgrad_bf16_partial(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ x2, int Ca,
    const __nv_bfloat16* __restrict__ dy, float* __restrict__ part, int N, int H, int W, int Cin,
    int Cout, long long chunk, int S, int u) {
  const int CG = Cin / 8;
  const long long E8 = (long long)Cout * 9 * CG;  // 8-wide output groups
  const int Ho = (H - 1) / u + 1, Wo = (W - 1) / u + 1;
  const long long P = (long long)N * Ho * Wo;     // dy's pixels
  const int split = blockIdx.y;
  const long long p0 = split * chunk;
  const long long p1 = p0 + chunk < P ? p0 + chunk : P;
  const long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long dwsize = (long long)Cout * 9 * Cin;
  if (e < E8) {
    int c0 = (int)(e % CG) * 8;
    int t = (int)((e / CG) % 9);
    int k = (int)(e / (9LL * CG));
    int r = t / 3, s = t % 3;
    // channel-split input: this thread's 8 channels lie in one part
    const __nv_bfloat16* xs = c0 < Ca ? x + c0 : x2 + (c0 - Ca);
    const int xstride = c0 < Ca ? Ca : Cin - Ca;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (long long p = p0; p < p1; ++p) {
      const int wo = (int)(p % Wo), ho = (int)((p / Wo) % Ho);
      const long long n = p / ((long long)Wo * Ho);
      int hi = u * ho + r - 1, wi = u * wo + s - 1;
      if (hi < 0 || hi >= H || wi < 0 || wi >= W) continue;
      float d = __bfloat162float(dy[p * Cout + k]);
      float xf[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(xs + ((n * H + hi) * W + wi) * xstride)), xf);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(d, xf[i], acc[i]);
    }
    float* o = part + (long long)split * dwsize + ((long long)k * 9 + t) * Cin + c0;
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = acc[i];
  }
  if (blockIdx.x == 0) {
    for (int k = threadIdx.x; k < Cout; k += blockDim.x) {
      float acc = 0.0f;
      for (long long p = p0; p < p1; ++p) acc += __bfloat162float(dy[p * Cout + k]);
      part[(long long)S * dwsize + (long long)split * Cout + k] = acc;
    }
  }
}

// wgrad partial sums, Cin == 8: one block per (split, 128-channel slice of
// Cout).  Thread (k, half): half 0 sums taps 0..4, half 1 taps 5..8 (8
// channels each) for output channel k; half 0 also sums dbias.
__global__ void __launch_bounds__(kThreads) k_wgrad_bf16_c8_partial(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ dy,
    float* __restrict__ part, int N, int H, int W, int Cout, long long chunk, int S) {
  const long long P = (long long)N * H * W;
  const int split = blockIdx.y;
  const long long p0 = split * chunk;
  const long long p1 = p0 + chunk < P ? p0 + chunk : P;
  const int k = blockIdx.x * 128 + (threadIdx.x & 127);
  const int half = threadIdx.x >> 7;
  const int t0 = half ? 5 : 0, nt = half ? 4 : 5;
  const bool active = k < Cout;
  float acc[5][8];
  float dbacc = 0.0f;
#pragma unroll
  for (int j = 0; j < 5; ++j)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[j][i] = 0.0f;
  if (active) {
#pragma unroll 1
    for (long long p = p0; p < p1; ++p) {
      int ww = (int)(p % W), hh = (int)((p / W) % H);
      float d = __bfloat162float(dy[p * Cout + k]);
      dbacc += d;
#pragma unroll
      for (int j = 0; j < 5; ++j) {
        if (j < nt) {
          int t = t0 + j, r = t / 3, s = t % 3;
          int hi = hh + r - 1, wi = ww + s - 1;
          if (hi >= 0 && hi < H && wi >= 0 && wi < W) {
            float xf[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(x + (p + (long long)(r - 1) * W + (s - 1)) * 8)), xf);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[j][i] = fmaf(d, xf[i], acc[j][i]);
          }
        }
      }
    }
    const long long dwsize = (long long)Cout * 72;
    float* o = part + (long long)split * dwsize + (long long)k * 72;
#pragma unroll
    for (int j = 0; j < 5; ++j)
      if (j < nt) {
        float4* o4 = reinterpret_cast<float4*>(o + (t0 + j) * 8);
        o4[0] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
        o4[1] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
      }
    if (half == 0) part[(long long)S * dwsize + (long long)split * Cout + k] = dbacc;
  }
}

// The split counts of one reduction: the partials hold Sreg slices of dw, then
// Sreg rows of dbias; output channels below k1 (dw rows, and dbias entries)
// have S1 valid splits, the others S2 (a weight gradient computed in two
// parts with two split plans; k1 = Cout when there is one).
struct RedSplits {
  int Sreg, S1, S2, k1;
};

// dw[e] = sum_{s=0}^{S-1} part[s][e] in increasing s (four partials loaded at a
// time, added strictly in order), four elements per thread; dbias likewise
// over its partial rows stored after the Sreg dw slices.  For layers whose
// split count is small (a few partials of a large dw).
__global__ void k_wgrad_reduce(const float* __restrict__ part, float* __restrict__ dw,
                               float* __restrict__ db, long long dwsize, int Cout, RedSplits rs) {
  pdl_trigger();
  pdl_wait();  // the partials of the kernel before
  const long long n4 = dwsize / 4;
  const long long n1 = (long long)rs.k1 * (dwsize / Cout) / 4;  // float4 columns of rows < k1
  const long long total = n4 + Cout;
  const float4* p4 = reinterpret_cast<const float4*>(part);
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    if (e < n4) {
      const int S = e < n1 ? rs.S1 : rs.S2;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      int s = 0;
      for (; s + 4 <= S; s += 4) {
        const float4 a0 = __ldg(p4 + (long long)s * n4 + e);
        const float4 a1 = __ldg(p4 + (long long)(s + 1) * n4 + e);
        const float4 a2 = __ldg(p4 + (long long)(s + 2) * n4 + e);
        const float4 a3 = __ldg(p4 + (long long)(s + 3) * n4 + e);
        acc.x += a0.x; acc.y += a0.y; acc.z += a0.z; acc.w += a0.w;
        acc.x += a1.x; acc.y += a1.y; acc.z += a1.z; acc.w += a1.w;
        acc.x += a2.x; acc.y += a2.y; acc.z += a2.z; acc.w += a2.w;
        acc.x += a3.x; acc.y += a3.y; acc.z += a3.z; acc.w += a3.w;
      }
      for (; s < S; ++s) {
        const float4 a = __ldg(p4 + (long long)s * n4 + e);
        acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
      }
      reinterpret_cast<float4*>(dw)[e] = acc;
    } else if (db) {
      const long long k = e - n4;
      const int S = k < rs.k1 ? rs.S1 : rs.S2;
      float acc = 0.0f;
      for (int s = 0; s < S; ++s) acc += part[(long long)rs.Sreg * dwsize + (long long)s * Cout + k];
      db[k] = acc;
    }
  }
}

// The same sum for wide splits (a layer with few output tiles has up to
// hundreds of splits of a small dw), in another fixed order: split group
// g = 0..G-1 (in order) of the sums over s = g, g + G, g + 2G, ... (each in
// increasing s).  A block of 256 threads covers 256 / G float4 columns with G
// split groups, so the splits are read by G thread rows at once instead of one
// thread per column walking all of them.  G is 8, or 32 when the columns are
// too few to give every SM two blocks of 32 columns (a small dw such as the
// 8-channel stem's: 32 groups of 8 columns, four times the blocks and a
// quarter of the loads per thread).  The order depends only on the shape and
// S, never on timing, and the result is bit-identical run to run.  dbias rides
// along as Cout / 4 more float4 columns over its Sdb partial rows stored after
// the S dw slices.
constexpr int kRedThreads = 256;

template <int G>
__global__ void __launch_bounds__(kRedThreads)
    k_wgrad_reduce_wide(const float* __restrict__ part, float* __restrict__ dw, float* __restrict__ db,
                        long long dwsize, int Cout, RedSplits rs) {
  constexpr int CW = kRedThreads / G;  // float4 columns per block
  __shared__ float4 red[G][CW];
  pdl_trigger();
  pdl_wait();  // the partials of the kernel before
  const int x = threadIdx.x, g = threadIdx.y;
  const long long n4 = dwsize / 4;
  const long long n1 = (long long)rs.k1 * (dwsize / Cout) / 4;  // float4 columns of rows < k1
  const long long col = blockIdx.x * (long long)CW + x;
  const bool bias_col = col >= n4;
  const long long total = n4 + (db ? Cout / 4 : 0);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col < total) {
    const float4* src = reinterpret_cast<const float4*>(bias_col ? part + (long long)rs.Sreg * dwsize : part);
    const long long c = bias_col ? col - n4 : col;
    const long long stride = bias_col ? Cout / 4 : n4;
    const int n = (bias_col ? 4 * c < rs.k1 : c < n1) ? rs.S1 : rs.S2;
#pragma unroll 4
    for (int sp = g; sp < n; sp += G) {
      const float4 a = __ldg(src + (long long)sp * stride + c);
      acc.x += a.x;
      acc.y += a.y;
      acc.z += a.z;
      acc.w += a.w;
    }
  }
  red[g][x] = acc;
  __syncthreads();
  if (g == 0 && col < total) {
    float4 t = red[0][x];
#pragma unroll
    for (int i = 1; i < G; ++i) {
      const float4 a = red[i][x];
      t.x += a.x;
      t.y += a.y;
      t.z += a.z;
      t.w += a.w;
    }
    if (bias_col) {  // dbias need only be 4-byte aligned: scalar stores
      float* o = db + (col - n4) * 4;
      o[0] = t.x;
      o[1] = t.y;
      o[2] = t.z;
      o[3] = t.w;
    } else {
      reinterpret_cast<float4*>(dw)[col] = t;
    }
  }
}

int grid_for(long long work, int per_block = kThreads) {
  long long g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > 65535LL * 16) g = 65535LL * 16;
  return (int)g;
}

int launch_status() {
  return cudaGetLastError() == cudaSuccess ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

struct WgradPlan {
  int S;
  long long chunk;
  bool c8;
};

WgradPlan wgrad_plan(const Shape& s) {
  WgradPlan pl;
  const long long P = s.Po();  // splits run over dy's pixels
  pl.c8 = (s.Cin == 8 && s.u == 1);
  long long blocks_per_split;
  if (pl.c8) {
    blocks_per_split = (s.Cout + 127) / 128;
  } else {
    long long E8 = (long long)s.Cout * 9 * (s.Cin / 8);
    blocks_per_split = (E8 + kThreads - 1) / kThreads;
  }
  long long target = 4LL * kPlanSms;  // blocks in flight across the device
  long long S = (target + blocks_per_split - 1) / blocks_per_split;
  if (S < 1) S = 1;
  if (S > P) S = P;
  if (S > 65535) S = 65535;
  pl.chunk = (P + S - 1) / S;
  pl.S = (int)((P + pl.chunk - 1) / pl.chunk);
  return pl;
}

}  // namespace

// Partial sums of S splits -> dw, dbias.  Which fixed summation order is used
// depends only on S: per column in split order below kWideSplits splits,
// eight split groups per column from there on.
constexpr int kWideSplits = 16;

int launch_wgrad_reduce2(const float* part, float* dw, float* db, long long dwsize, int Cout, int Sreg,
                         int S1, int S2, int k1, cudaStream_t st) {
  const RedSplits rs{Sreg, S1, S2, k1};
  if ((S1 > S2 ? S1 : S2) >= kWideSplits) {
    const long long cols = dwsize / 4 + (db ? Cout / 4 : 0);
    if (cols < 2LL * kPlanSms * 32)
      launch_pdl(k_wgrad_reduce_wide<32>, dim3((unsigned)((cols + 7) / 8)), dim3(8, 32), 0, st, part,
                 dw, db, dwsize, Cout, rs);
    else
      launch_pdl(k_wgrad_reduce_wide<8>, dim3((unsigned)((cols + 31) / 32)), dim3(32, 8), 0, st, part,
                 dw, db, dwsize, Cout, rs);
  } else {
    launch_pdl(k_wgrad_reduce, dim3(grid_for(dwsize / 4 + Cout)), dim3(kThreads), 0, st, part, dw, db,
               dwsize, Cout, rs);
  }
  return launch_status();
}

int launch_wgrad_reduce(const float* part, float* dw, float* db, long long dwsize, int Cout, int S,
                        int Sdb, cudaStream_t st) {
  (void)Sdb;  // dbias has as many partial rows as dw has slices
  return launch_wgrad_reduce2(part, dw, db, dwsize, Cout, S, S, S, Cout, st);
}

// ---------------------------------------------------------------- launchers
int simt_fwd_f32(const float* x, const float* w, const float* bias, float* y, const Shape& s,
                 int act, cudaStream_t st) {
  long long total = s.P() * s.Cout;
  k_fwd_f32<<<grid_for(total), kThreads, 0, st>>>(x, w, bias, y, s.N, s.H, s.W, s.Cin, s.Cout, act);
  return launch_status();
}

int simt_dgrad_f32(const float* dy, const float* w, float* dx, const Shape& s, cudaStream_t st) {
  long long total = s.P() * s.Cin;
  k_dgrad_f32<<<grid_for(total), kThreads, 0, st>>>(dy, w, dx, s.N, s.H, s.W, s.Cin, s.Cout);
  return launch_status();
}

int simt_wgrad_f32(const float* x, const float* dy, float* dw, float* db, const Shape& s,
                   cudaStream_t st) {
  long long total = (long long)s.Cout * 9 * s.Cin;
  k_wgrad_f32<<<grid_for(total), kThreads, 0, st>>>(x, dy, dw, db, s.N, s.H, s.W, s.Cin, s.Cout);
  return launch_status();
}

int simt_fwd_bf16(const void* x, const void* w, const float* bias, void* y, const Shape& s,
                  int act, int out_f32, const EpiExtra& ex, const CatSplit& cat, cudaStream_t st) {
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  const __nv_bfloat16* wb = static_cast<const __nv_bfloat16*>(w);
  __nv_bfloat16* zb = static_cast<__nv_bfloat16*>(ex.zout);
  if (s.Cin == 8 && s.Cout <= 512 && !cat.on() && s.u == 1) {
    size_t sm = (size_t)s.Cout * 72 * sizeof(float);
    if (sm > 48 * 1024 &&
        cudaFuncSetAttribute(k_fwd_bf16_c8, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) !=
            cudaSuccess)
      return CONV3X3_ERR_CUDA;
    k_fwd_bf16_c8<<<grid_for(s.P()), kThreads, sm, st>>>(xb, wb, bias, y, zb, s.N, s.H, s.W,
                                                         s.Cout, act, out_f32);
  } else {
    k_fwd_bf16_gen<<<grid_for(s.Po() * (s.Cout / 8)), kThreads, 0, st>>>(
        xb, static_cast<const __nv_bfloat16*>(cat.b), cat.on() ? cat.Ca : s.Cin, wb, bias, y, zb,
        s.N, s.H, s.W, s.Cin, s.Cout, act, out_f32, s.u);
  }
  return launch_status();
}

int simt_dgrad_bf16(const void* dy, const void* w, void* dx, const Shape& s, int out_f32,
                    const EpiExtra& ex, const CatSplit& cat, cudaStream_t st) {
  const __nv_bfloat16* db = static_cast<const __nv_bfloat16*>(dy);
  const __nv_bfloat16* wb = static_cast<const __nv_bfloat16*>(w);
  const __nv_bfloat16* zb = static_cast<const __nv_bfloat16*>(ex.zin);
  if (s.Cin == 8 && s.Cout <= 512 && !cat.on() && s.u == 1) {
    size_t sm = (size_t)s.Cout * 72 * sizeof(float);
    if (sm > 48 * 1024 &&
        cudaFuncSetAttribute(k_dgrad_bf16_c8, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm) != cudaSuccess)
      return CONV3X3_ERR_CUDA;
    k_dgrad_bf16_c8<<<grid_for(s.P()), kThreads, sm, st>>>(db, wb, dx, zb, ex.zin_act, s.N, s.H,
                                                           s.W, s.Cout, out_f32);
  } else {
    k_dgrad_bf16_gen<<<grid_for(s.P() * (s.Cin / 8)), kThreads, 0, st>>>(
        db, wb, dx, cat.b, cat.on() ? cat.Ca : s.Cin, zb,
        static_cast<const __nv_bfloat16*>(ex.zin_b), ex.zin_act, s.N, s.H, s.W, s.Cin, s.Cout,
        out_f32, s.u);
  }
  return launch_status();
}

size_t simt_wgrad_workspace(const Shape& s, int /*num_sms*/) {
  WgradPlan pl = wgrad_plan(s);
  long long dwsize = (long long)s.Cout * 9 * s.Cin;
  return (size_t)pl.S * (size_t)(dwsize + s.Cout) * sizeof(float);
}

int simt_wgrad_bf16(const void* x, const void* dy, float* dw, float* db, const Shape& s,
                    void* ws, size_t ws_bytes, int num_sms, const CatSplit& cat, cudaStream_t st) {
  if (ws_bytes < simt_wgrad_workspace(s, num_sms) || ws == nullptr) return CONV3X3_ERR_WORKSPACE;
  WgradPlan pl = wgrad_plan(s);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  const __nv_bfloat16* dyb = static_cast<const __nv_bfloat16*>(dy);
  float* part = static_cast<float*>(ws);
  if (pl.c8) {
    dim3 grid((s.Cout + 127) / 128, pl.S);
    k_wgrad_bf16_c8_partial<<<grid, kThreads, 0, st>>>(xb, dyb, part, s.N, s.H, s.W, s.Cout,
                                                       pl.chunk, pl.S);
  } else {
    long long E8 = (long long)s.Cout * 9 * (s.Cin / 8);
    dim3 grid((unsigned)((E8 + kThreads - 1) / kThreads), pl.S);
    k_wgrad_bf16_partial<<<grid, kThreads, 0, st>>>(
        xb, static_cast<const __nv_bfloat16*>(cat.b), cat.on() ? cat.Ca : s.Cin, dyb, part, s.N,
        s.H, s.W, s.Cin, s.Cout, pl.chunk, pl.S, s.u);
  }
  if (cudaGetLastError() != cudaSuccess) return CONV3X3_ERR_CUDA;
  long long dwsize = (long long)s.Cout * 9 * s.Cin;
  return launch_wgrad_reduce(part, dw, db, dwsize, s.Cout, pl.S, pl.S, st);
}

}  // namespace c3
