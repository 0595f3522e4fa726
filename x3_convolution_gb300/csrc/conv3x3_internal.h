// conv3x3_internal.h -- declarations shared by the library's translation units
// (host launchers of each kernel family).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/conv3x3.h"

namespace c3 {

// Problem shape as the host dispatcher sees it.
struct Shape {
  int N, Cin, Cout, H, W;  // H, W: the input's (x's, dx's) grid
  int u = 1;               // stride: 1, or 2 for a downsampling conv (pad 1 either way)
  long long P() const { return (long long)N * H * W; }
  int Ho() const { return (H - 1) / u + 1; }  // output (y's, dy's) grid
  int Wo() const { return (W - 1) / u + 1; }
  long long Po() const { return (long long)N * Ho() * Wo(); }
};

// Programmatic dependent launch.  The tensor-path kernels start with
// pdl_trigger() (their dependents may begin launching; the wgrad mainloops
// skip it, see there) and execute pdl_wait() -- which returns once the previous
// kernel in the stream has completed and its writes are visible -- before
// their first access to global memory, so only set-up (barrier init, TMEM
// allocation, descriptor prefetch) overlaps the previous kernel's tail.
// Launched without the attribute, both are no-ops.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Whether launches carry the programmatic-serialization attribute
// (CONV3X3_PDL=0 turns it off).
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Per-call device context: status word and wait bound.
struct DevCtx {
  unsigned* status;          // device address of the status word
  unsigned long long wait_ns;  // bound on every device-side wait
  int num_sms;
  int device;
};

// Optional extras of the fused epilogue (bf16 tensors laid out like the output):
// zout -- forward also stores z = conv + bias before the activation;
// zin  -- dgrad scales its result by act'(zin) for zin_act.
struct EpiExtra {
  void* zout = nullptr;
  const void* zin = nullptr;
  const void* zin_b = nullptr;  // z_in of channels [Ca, Cin) when the input is split (CatSplit)
  int zin_act = CONV3X3_ACT_NONE;
};

// A channel-split input (fwd, wgrad) or input gradient (dgrad): channels
// [0, Ca) live in the primary tensor ([P][Ca]), channels [Ca, Cin) in `b`
// ([P][Cin - Ca]).  b == nullptr: one tensor of Cin channels.
struct CatSplit {
  void* b = nullptr;
  int Ca = 0;
  bool on() const { return b != nullptr; }
};

// ---- CUDA-core kernels (simt.cu) ----
int simt_fwd_f32(const float* x, const float* w, const float* bias, float* y, const Shape& s,
                 int act, cudaStream_t st);
int simt_dgrad_f32(const float* dy, const float* w, float* dx, const Shape& s, cudaStream_t st);
int simt_wgrad_f32(const float* x, const float* dy, float* dw, float* db, const Shape& s,
                   cudaStream_t st);

int simt_fwd_bf16(const void* x, const void* w, const float* bias, void* y, const Shape& s,
                  int act, int out_f32, const EpiExtra& ex, const CatSplit& cat, cudaStream_t st);
int simt_dgrad_bf16(const void* dy, const void* w, void* dx, const Shape& s, int out_f32,
                    const EpiExtra& ex, const CatSplit& cat, cudaStream_t st);
size_t simt_wgrad_workspace(const Shape& s, int num_sms);
int simt_wgrad_bf16(const void* x, const void* dy, float* dw, float* db, const Shape& s,
                    void* ws, size_t ws_bytes, int num_sms, const CatSplit& cat, cudaStream_t st);

// ---- tensor-core kernels (tc.cu) ----
bool tc_supported(int pass, const Shape& s);
bool tc_supports_cat(const Shape& s, const CatSplit& cat);
int tc_fwd(const void* x, const void* w, const float* bias, void* y, const Shape& s, int act,
           int out_f32, const EpiExtra& ex, const CatSplit& cat, const DevCtx& d, cudaStream_t st);
int tc_dgrad(const void* dy, const void* w, void* dx, const Shape& s, int out_f32,
             const EpiExtra& ex, const CatSplit& cat, const DevCtx& d, cudaStream_t st);
size_t tc_wgrad_workspace(const Shape& s, int num_sms);
int tc_wgrad(const void* x, const void* dy, float* dw, float* db, const Shape& s, void* ws,
             size_t ws_bytes, const CatSplit& cat, const DevCtx& d, cudaStream_t st);

// ---- driver entry points (api.cu) ----
typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*PFN_encodeIm2col)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                     const cuuint64_t*, const cuuint64_t*, const int*, const int*,
                                     cuuint32_t, cuuint32_t, const cuuint32_t*,
                                     CUtensorMapInterleave, CUtensorMapSwizzle,
                                     CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
PFN_encodeTiled encode_tiled_fn();
PFN_encodeIm2col encode_im2col_fn();

}  // namespace c3
