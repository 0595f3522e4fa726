/*
 * conv3x3.h -- C ABI of libconv3x3.so: stride-1, zero-pad-1 3x3 convolution
 * forward, input gradient (dgrad) and weight gradient (wgrad) on one GB300
 * (sm_103a).
 *
 * The operation is the 3x3 convolution that the subject page's custom CUDA
 * kernels compute, forward and backward, inside a diffusion UNet training step
 * (clu0's C++/CUDA UNet diffusion, sourcepulse.org project page, "How It Works"
 * and "Highlighted Details").  The page does not write it down; this library
 * computes the PyTorch Conv2d cross-correlation (no kernel flip) with stride 1,
 * padding 1, dilation 1, groups 1:
 *
 *   fwd    z[n,h,w,k]  = bias[k] + sum_{r,s,c} x[n,h+r-1,w+s-1,c] * w[k,r,s,c]
 *          y = z (act NONE), z * sigmoid(z) (act SILU) or
 *          max(z, 0.2 z) (act LRELU)
 *   dgrad  dx[n,h,w,c] = sum_{r,s,k} dy[n,h+1-r,w+1-s,k] * w[k,r,s,c]
 *   wgrad  dw[k,r,s,c] = sum_{n,h,w} dy[n,h,w,k] * x[n,h+r-1,w+s-1,c]
 *          dbias[k]    = sum_{n,h,w} dy[n,h,w,k]
 *
 * Taps outside the image read zero.  dy is the gradient with respect to the
 * pre-activation z (the SiLU backward, if any, is the caller's step).
 *
 * Layouts (all dense, no padding between rows):
 *   activations x, y, dx, dy : NHWC, c fastest       ([N][H][W][C])
 *   weights w, dw             : KRSC = [Cout][3][3][Cin], c fastest
 *   bias, dbias               : [Cout]
 * Element types: the production entry points take bf16 activations and
 * weights, fp32 bias, fp32 dw / dbias, and accumulate in fp32.  The *_f32
 * entry points take fp32 everywhere and accumulate with fp32 FMA on CUDA cores
 * (never TF32).
 *
 * Ownership: the caller allocates every device buffer (inputs, outputs and the
 * wgrad workspace) and keeps it alive until the work on `stream` completes.
 * The library allocates no device memory; it keeps only host-side state (a
 * driver entry point, per-device attributes) and one device status word.
 *
 * Asynchrony: every call enqueues work on `stream` (a cudaStream_t passed as
 * void*, NULL = legacy default stream) and returns without synchronising.
 *
 * Errors: every call returns a conv3x3_status; nothing is thrown across the ABI.
 * Arguments are validated on the host before anything is launched:
 *   - N, H, W >= 1; Cin, Cout >= 8 and multiples of 8;
 *   - every pointer non-NULL (bias / dbias may be NULL) and 16-byte aligned;
 *   - N*H*W*max(Cin,Cout) < 2^31 elements per activation tensor, H, W <= 65535;
 *   - act in {NONE, SILU, LRELU}; out_dtype in {BF16, F32}; path in {AUTO, TENSOR, SIMT}.
 * A launch failure returns CONV3X3_ERR_CUDA.  The library keeps per-device
 * state for device ordinals 0..63; a call made with a higher ordinal current
 * returns CONV3X3_ERR_UNSUPPORTED.  Kernels that wait on the
 * hardware (mbarrier / TMA / tensor-core completion) give up after a bounded
 * time, record CONV3X3_ERR_TIMEOUT in the device status word and exit cleanly;
 * read it with conv3x3_device_status().  The bound is 2 s per wait
 * (CONV3X3_WAIT_LIMIT_NS, read once per process), timed on the global
 * nanosecond timer and also required to have passed on the SM cycle counter
 * (bound / 2 cycles).
 *
 * Tuning override: the environment variable CONV3X3_TILE forces the forward /
 * dgrad tensor-core tile: "<BN>x<MT>" (BN in {64,128,192,256}, MT in {1,2},
 * 2*MT*BN <= 512) selects the im2col kernel with MT*128 pixels x BN channels,
 * "halo<BN>" (BN in {64,128}; images of width 16, 32 or 64 whose height is a
 * multiple of 256/W) the row-halo kernel.  Unset, the library picks.
 * "128x2" runs transposed (weights as the M = 128 operand, 256 pixels as N) and
 * "128x2n" untransposed; "256x1" runs on two-CTA clusters (one 256-pixel x
 * 256-channel tile per pair, tcgen05 cta_group::2) and "256x1n" on one CTA;
 * "pair128", "pair192", "pair256", "pair384" run 256-pixel x 128/192/256/384-
 * channel tiles on two-CTA clusters.  CONV3X3_PAIR384=0 keeps 384-channel
 * outputs off the 384-wide two-CTA tile (unset: taken with at least six input
 * chunks and enough 256-pixel tiles to fill 3/8 of the GPU in one round).
 * CONV3X3_PKS=0|1 forbids (or, where the shape allows, forces) 256-pixel x
 * 256-channel two-CTA tiles whose K is split over the two CTA pairs of a
 * cluster of four and summed through distributed shared memory (outputs a
 * multiple of 256, an even input chunk count of at least four; unset: taken
 * with at least eight input chunks where whole pair tiles would fill under
 * half of the GPU but such clusters fill at least half of it, as on 8x8
 * layers of 512 channels).
 * CONV3X3_KSPLIT=0|1 forces (or forbids) 128 x 256 tiles whose K is split over
 * a two-CTA cluster and summed through distributed shared memory (outputs a
 * multiple of 256 channels; unset: where such tiles fill a quarter to all of
 * the GPU in pairs and the input has at least 1024 channels).
 * CONV3X3_PAIR=0|1 forces the two-CTA choice for 256-channel tiles (unset: dgrad
 * and forwards of at least 256 input channels, with two rounds of pair tiles).
 * CONV3X3_KC=1|2 forces the 64-channel chunks per pipeline stage of the im2col
 * kernel (2 for 128x1 tiles unless set); CONV3X3_PAIR_KC=1 keeps one chunk per
 * stage in the 256-channel two-CTA tiles (unset: two where the input channels
 * are a whole number of 128).  CONV3X3_PAIR_HALF=0 keeps whole 256-channel
 * two-CTA tiles in a last round that fills at most half of the pairs (unset:
 * that round's tiles run as two 128-channel halves each); =all splits every
 * such tile (tests).  CONV3X3_WGRAD_SPLITS=<S> forces the
 * weight gradient's split count (set it before querying the workspace size).
 * CONV3X3_WGRAD_ROWS=0|1 chooses how the weight gradient stages x: im2col
 * boxes per tap (0), or one zero-padded box per image row that all three taps
 * of a kernel row read (1; stride 1, width 16, 32 or 64).  Unset: the latter
 * for width 64 only.  CONV3X3_WGRAD_PAIR=0 keeps the weight gradient of Cout a
 * multiple of 256 on one-CTA tiles (by default, where x is staged as im2col
 * boxes, it runs on two-CTA clusters with 256-output-channel tiles; the
 * workspace size covers either).  CONV3X3_WGRAD_HYBRID=0|1 forbids (or forces,
 * wherever it applies) the split of a Cout above 256 that is not a multiple of
 * 256 into two-CTA tiles over its first 256 k channels and one-CTA tiles over
 * the rest, two launches with one workspace and one reduction (unset: where
 * the one-CTA plan would leave over a quarter of the SMs idle).
 * CONV3X3_WGRAD_PART_TMA=0 makes the weight gradient write its split partials
 * with per-thread stores instead of TMA tensor stores (at least 32 input
 * channels).  CONV3X3_EPI_TMA=0 makes forward and input-gradient tiles store
 * their output from each thread instead of through TMA tensor stores (taken
 * for one plain bf16 output: on every tile where every CTA or CTA pair has
 * one, else on each CTA's or pair's last tile); CONV3X3_EPI_TMA=1 keeps them
 * to one-tile launches.
 * CONV3X3_STEM_ZTMA=0 makes the 8-input-channel forward that also stores z
 * store y and z from each thread instead of through TMA tensor stores (taken
 * with row staging, bf16 y and at most 128 output channels).
 * CONV3X3_STEM_ROWS=0 makes the 8-input-channel forward
 * and weight gradient stage x as im2col boxes even where they would stage
 * whole image rows (forward: widths 32 and 64; weight gradient: width 64,
 * three column-shifted copies of three zero-padded image rows per 64-pixel
 * k-block).
 * CONV3X3_STEM_DGRAD=rows runs the 8-output-channel input gradient of width 64
 * as row bands instead of tiles.
 * CONV3X3_PDL=0 launches without programmatic dependent launch (by default a
 * kernel's set-up overlaps the end of the previous kernel in the stream; each
 * kernel still waits for that kernel to complete before touching memory).
 * These variables are read when a call is made (CONV3X3_PDL once per process).
 */
#ifndef CONV3X3_H
#define CONV3X3_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CONV3X3_OK = 0,
  CONV3X3_ERR_INVALID_ARG = 1, /* bad shape, pointer, alignment or enum      */
  CONV3X3_ERR_UNSUPPORTED = 2, /* valid arguments this build cannot run      */
  CONV3X3_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed        */
  CONV3X3_ERR_TIMEOUT = 4,     /* a device-side wait hit its bound           */
  CONV3X3_ERR_WORKSPACE = 5    /* wgrad workspace missing or too small       */
} conv3x3_status;

/* Epilogue activations: none; SiLU z*sigmoid(z); leaky ReLU, z for z >= 0 and
 * 0.2 z below.  The last is the bias + leaky ReLU fused op of the StyleGAN2
 * custom-kernel blog (page titled "Dim3 grid calculation code", opening
 * paragraphs on the two custom kernels).  That page gives no slope and no gain:
 * the slope is taken as 0.2 and no output gain is applied. */
enum { CONV3X3_ACT_NONE = 0, CONV3X3_ACT_SILU = 1, CONV3X3_ACT_LRELU = 2 };
enum { CONV3X3_DT_BF16 = 0, CONV3X3_DT_F32 = 1 };
/* Kernel family: AUTO picks per shape; TENSOR = TMA-im2col + tcgen05/TMEM
 * implicit GEMM; SIMT = CUDA-core fp32-FMA kernels with 128-bit loads. */
enum { CONV3X3_PATH_AUTO = 0, CONV3X3_PATH_TENSOR = 1, CONV3X3_PATH_SIMT = 2 };

/* Forward with fused bias + activation epilogue.
 * x [N][H][W][Cin] bf16, w [Cout][3][3][Cin] bf16, bias [Cout] fp32 or NULL,
 * y [N][H][W][Cout] bf16 (written, round-to-nearest-even from the fp32 result). */
int conv3x3_fwd(const void* x, const void* w, const float* bias, void* y,
                int N, int Cin, int Cout, int H, int W, int act, void* stream);

/* Input gradient.  dy [N][H][W][Cout] bf16, w [Cout][3][3][Cin] bf16,
 * dx [N][H][W][Cin] bf16 (written). */
int conv3x3_dgrad(const void* dy, const void* w, void* dx,
                  int N, int Cin, int Cout, int H, int W, void* stream);

/* Weight and bias gradient.  x [N][H][W][Cin] bf16, dy [N][H][W][Cout] bf16,
 * dw [Cout][3][3][Cin] fp32 (overwritten, not accumulated), dbias [Cout] fp32
 * or NULL (overwritten).  The cross-CTA reduction sums fixed partial slices in
 * a fixed order, so repeated calls give bit-identical dw and dbias.
 * `workspace` is caller-owned device scratch of at least
 * conv3x3_wgrad_workspace_bytes(...) bytes (may be NULL when that is 0),
 * 256-byte aligned; its contents on entry do not matter. */
int conv3x3_wgrad(const void* x, const void* dy, float* dw, float* dbias,
                  int N, int Cin, int Cout, int H, int W,
                  void* workspace, size_t workspace_bytes, void* stream);

/* Scratch bytes conv3x3_wgrad needs for this shape (0 for invalid shapes).
 * Pure host computation; needs no GPU. */
size_t conv3x3_wgrad_workspace_bytes(int N, int Cin, int Cout, int H, int W);

/* Parity / dispatch variants of the same kernels.
 * out_dtype = CONV3X3_DT_F32 writes the fp32 epilogue result before the bf16
 * rounding (y or dx is then an fp32 buffer); `path` forces a kernel family.
 * CONV3X3_ERR_UNSUPPORTED if the forced family cannot run the shape. */
int conv3x3_fwd_ex(const void* x, const void* w, const float* bias, void* y,
                   int N, int Cin, int Cout, int H, int W, int act,
                   int out_dtype, int path, void* stream);
int conv3x3_dgrad_ex(const void* dy, const void* w, void* dx,
                     int N, int Cin, int Cout, int H, int W,
                     int out_dtype, int path, void* stream);
int conv3x3_wgrad_ex(const void* x, const void* dy, float* dw, float* dbias,
                     int N, int Cin, int Cout, int H, int W,
                     void* workspace, size_t workspace_bytes, int path, void* stream);
size_t conv3x3_wgrad_workspace_bytes_ex(int N, int Cin, int Cout, int H, int W, int path);

/* Backward through a layer's activation, fused into the convolutions' own
 * epilogues.  The subject page (clu0's C++/CUDA UNet diffusion, sourcepulse.org
 * project page, "How It Works") puts the emphasis on minimising memory
 * transfers; these two calls remove the elementwise pass dz = dy * act'(z)
 * that a training step otherwise runs between the convolutions.
 *
 * conv3x3_fwd_save_z: conv3x3_fwd_ex, and also stores the pre-activation
 *   z = conv + bias, rounded once to bf16, in z [N][H][W][Cout] (16-byte
 *   aligned; it must not overlap y).  y = act(z) is computed from the fp32 z,
 *   exactly as conv3x3_fwd_ex computes it.
 * conv3x3_dgrad_act: the input gradient of a convolution whose input was
 *   x = act_in(z_in):  dx = act_in'(z_in) * dgrad(dy, w), the product taken in
 *   fp32 on the accumulator and rounded once.  z_in [N][H][W][Cin] bf16,
 *   16-byte aligned, must not overlap dx.  act_in' is SiLU' = s (1 + z (1 - s))
 *   with s the logistic sigmoid, or leaky ReLU' = 1 for z > 0 and 0.2 for
 *   z <= 0; act_in = CONV3X3_ACT_NONE is plain dgrad and z_in is ignored (may be
 *   NULL).  The result is the gradient with respect to z_in: it feeds the
 *   previous layer's conv3x3_wgrad and conv3x3_dgrad_act directly.
 * Errors as conv3x3_fwd_ex / conv3x3_dgrad_ex, and CONV3X3_ERR_INVALID_ARG for
 * a missing, misaligned or overlapping z / z_in or an unknown act_in. */
int conv3x3_fwd_save_z(const void* x, const void* w, const float* bias, void* y, void* z,
                       int N, int Cin, int Cout, int H, int W, int act,
                       int out_dtype, int path, void* stream);
int conv3x3_dgrad_act(const void* dy, const void* w, const void* z_in, int act_in, void* dx,
                      int N, int Cin, int Cout, int H, int W,
                      int out_dtype, int path, void* stream);

/* fp32 check path: every tensor fp32 (same layouts), fp32 FMA on CUDA cores,
 * never TF32.  Any Cin, Cout >= 1; pointers 4-byte aligned.  wgrad needs no
 * workspace (pass NULL, 0). */
int conv3x3_fwd_f32(const float* x, const float* w, const float* bias, float* y,
                    int N, int Cin, int Cout, int H, int W, int act, void* stream);
int conv3x3_dgrad_f32(const float* dy, const float* w, float* dx,
                      int N, int Cin, int Cout, int H, int W, void* stream);
int conv3x3_wgrad_f32(const float* x, const float* dy, float* dw, float* dbias,
                      int N, int Cin, int Cout, int H, int W,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Reads and clears the current device's status word (CONV3X3_OK or
 * CONV3X3_ERR_TIMEOUT).  Synchronises `stream` first. */
int conv3x3_device_status(void* stream);

/* Self-test of the bounded-wait mechanism: launches one block that waits on an
 * mbarrier nobody arrives on, with a limit of `limit_ns` nanoseconds.  The
 * kernel gives up, records CONV3X3_ERR_TIMEOUT in the status word and returns;
 * the CUDA context stays usable.  Returns the launch status. */
int conv3x3_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

/* Weight gradient without caller-provided scratch.  The pages have no
 * counterpart of this entry point; it exists for callers that cannot allocate
 * device memory -- e.g. a plugin inside a host application whose memory pool
 * it may not draw on, or a latency-critical loop that may not call cudaMalloc
 * (which can synchronise the device) after start-up.
 * Same arguments, layouts and results as conv3x3_wgrad minus the workspace:
 * the split-K scratch is a fixed array of CONV3X3_WGRAD_NOALLOC_MAX_BYTES in
 * the library's own device memory, which every GPU that loads the library
 * holds until the process exits.  Allocates nothing.
 *   - Shapes whose conv3x3_wgrad_workspace_bytes() exceeds the maximum return
 *     CONV3X3_ERR_WORKSPACE before anything is launched; invalid shapes
 *     CONV3X3_ERR_INVALID_ARG.
 *   - The first call on a device looks up that device's copy of the array
 *     (cudaGetSymbolAddress, with the device current); make that first call
 *     before any stream capture.  Device ordinals 0..63 only (higher:
 *     CONV3X3_ERR_UNSUPPORTED).
 *   - All calls on a device share the array and it keeps the previous call's
 *     contents (nothing needs clearing: every partial read is written first).
 *     Calls whose work overlaps on the GPU -- different streams without an
 *     ordering between them -- race on the array; order them on one stream. */
#define CONV3X3_WGRAD_NOALLOC_MAX_BYTES (64ull << 20)
int conv3x3_wgrad_noalloc(const void* x, const void* dy, float* dw, float* dbias,
                          int N, int Cin, int Cout, int H, int W, void* stream);

/* Convolution of a channel-concatenated input without the concatenation.
 * A UNet (the architecture of the subject page, clu0's C++/CUDA UNet diffusion,
 * sourcepulse.org project page, "How It Works") feeds each up-path conv the
 * concatenation of its main branch and a skip from the down path.  These calls
 * take the two parts as separate tensors, so the concatenated copy is never
 * built (forward, weight gradient) and the input gradient comes back already
 * split (dgrad).  The results are those of the plain calls on
 * x = concat(xa, xb) along channels:
 *   xa [N][H][W][Ca], xb [N][H][W][Cin - Ca], both bf16, 16-byte aligned;
 *   w [Cout][3][3][Cin] (channels [0, Ca) act on xa, [Ca, Cin) on xb).
 *   0 < Ca < Cin, Ca a multiple of 8 (and of 64 for the tensor-core path:
 *   path = AUTO then falls back to the CUDA-core kernels, TENSOR returns
 *   CONV3X3_ERR_UNSUPPORTED).
 * conv3x3_fwd_cat:   as conv3x3_fwd_save_z; z may be NULL (no z stored).
 * conv3x3_dgrad_cat: dxa [N][H][W][Ca] and dxb [N][H][W][Cin - Ca] receive the
 *   two parts of dx (they must not overlap).  With act_in != NONE each part is
 *   scaled by act_in' of its pre-activation (za_in / zb_in, laid out like
 *   dxa / dxb), as conv3x3_dgrad_act does; with NONE both z pointers are ignored.
 * conv3x3_wgrad_cat: as conv3x3_wgrad_ex; the workspace size comes from
 *   conv3x3_wgrad_cat_workspace_bytes (0 for invalid arguments).
 * Errors as the plain calls, and CONV3X3_ERR_INVALID_ARG for a bad Ca, a
 * missing or misaligned part, or overlapping outputs. */
int conv3x3_fwd_cat(const void* xa, const void* xb, int Ca, const void* w, const float* bias,
                    void* y, void* z, int N, int Cin, int Cout, int H, int W, int act,
                    int out_dtype, int path, void* stream);
int conv3x3_dgrad_cat(const void* dy, const void* w, void* dxa, void* dxb, int Ca,
                      const void* za_in, const void* zb_in, int act_in,
                      int N, int Cin, int Cout, int H, int W, int out_dtype, int path,
                      void* stream);
int conv3x3_wgrad_cat(const void* xa, const void* xb, int Ca, const void* dy, float* dw,
                      float* dbias, int N, int Cin, int Cout, int H, int W,
                      void* workspace, size_t workspace_bytes, int path, void* stream);
size_t conv3x3_wgrad_cat_workspace_bytes(int N, int Cin, int Ca, int Cout, int H, int W,
                                         int path);

/* Strided (downsampling) convolution: the same 3x3 window and zero padding of
 * 1, moved `stride` input pixels per output pixel (stride 1 or 2).  The pages
 * reach downsampling only through the StyleGAN2 custom-kernel blog (page
 * titled "Dim3 grid calculation code", on up/downsampling); a UNet's down path
 * (the subject page's architecture) halves the resolution with a stride-2
 * 3x3 conv.  With Ho = (H - 1) / stride + 1 and Wo likewise:
 *   y[n,ho,wo,k] = act(b[k] + sum_{r,s,c} x[n, stride*ho + r - 1, stride*wo + s - 1, c] w[k,r,s,c])
 *   x, dx [N][H][W][Cin];  y, z, dy [N][Ho][Wo][Cout];  w KRSC as everywhere.
 * conv3x3_fwd_strided:   as conv3x3_fwd_save_z (z may be NULL).
 * conv3x3_dgrad_strided: dx = the adjoint of the forward applied to dy, scaled
 *   by act_in'(z_in) as in conv3x3_dgrad_act (act_in NONE: plain, z_in ignored).
 * conv3x3_wgrad_strided: as conv3x3_wgrad_ex; scratch size from
 *   conv3x3_wgrad_strided_workspace_bytes.
 * The tensor-core kernels take stride 2 when Cin >= 64 and Cout >= 64 (the
 * stride-2 dgrad runs as four output-parity classes with 1, 2, 2 and 4 taps);
 * other shapes use the CUDA-core kernels (path AUTO) or return
 * CONV3X3_ERR_UNSUPPORTED (path TENSOR).  Any other stride:
 * CONV3X3_ERR_INVALID_ARG. */
int conv3x3_fwd_strided(const void* x, const void* w, const float* bias, void* y, void* z,
                        int N, int Cin, int Cout, int H, int W, int stride, int act,
                        int out_dtype, int path, void* stream);
int conv3x3_dgrad_strided(const void* dy, const void* w, void* dx, const void* z_in, int act_in,
                          int N, int Cin, int Cout, int H, int W, int stride,
                          int out_dtype, int path, void* stream);
int conv3x3_wgrad_strided(const void* x, const void* dy, float* dw, float* dbias,
                          int N, int Cin, int Cout, int H, int W, int stride,
                          void* workspace, size_t workspace_bytes, int path, void* stream);
size_t conv3x3_wgrad_strided_workspace_bytes(int N, int Cin, int Cout, int H, int W, int stride,
                                             int path);

/* Static description of a status code ("ok", "invalid argument", ...). */
const char* conv3x3_status_string(int status);

/* Which kernel family `path = AUTO` picks for this shape and pass
 * (pass: 0 fwd, 1 dgrad, 2 wgrad).  Host-only. */
int conv3x3_auto_path(int pass, int N, int Cin, int Cout, int H, int W);

#ifdef __cplusplus
}
#endif

#endif /* CONV3X3_H */
