/*
 * upfirdn2d.h -- C ABI of the filtered up/downsampling op in libconv3x3.so.
 *
 * The operation is the one the StyleGAN2 custom-kernel blog (page titled
 * "Dim3 grid calculation code", first paragraph) describes: every channel of
 * every image goes through four steps, in this order,
 *   1. upsample: insert (up - 1) zeros after each pixel, along both axes;
 *   2. pad: pad_y0 / pad_y1 zero rows above / below, pad_x0 / pad_x1 zero
 *      columns left / right;
 *   3. FIR filter: 2-D convolution with the kh x kw kernel f (the kernel is
 *      flipped, as a convolution flips it), over the positions where it lies
 *      wholly inside the padded plane;
 *   4. downsample: keep every down-th pixel, starting with the first.
 * Written out for one output element:
 *   y[n,oy,ox,c] = sum_{a,b} f[a][b] * P[n, oy*down + kh-1-a, ox*down + kw-1-b, c]
 *   with P[n, p, q, c] = x[n, (p - pad_y0)/up, (q - pad_x0)/up, c] when both
 *   p - pad_y0 and q - pad_x0 are non-negative multiples of up inside the
 *   upsampled plane, and 0 otherwise;
 *   Ho = (H*up + pad_y0 + pad_y1 - kh) / down + 1, Wo likewise.
 * The page's own filter formula did not survive; a UNet's 2x resampling uses
 * the binomial [1,3,3,1] (x) [1,3,3,1] / 64 (times up^2 when upsampling, to
 * keep the mean), which the benchmark takes.  The gain is part of f.
 * The input gradient of upfirdn2d is upfirdn2d of dy with up and down swapped,
 * f flipped in both axes, and leading pads k - 1 - pad0 (the trailing pads
 * long enough to give back H x W).
 *
 * Layout: x [N][H][W][C] bf16 and y [N][Ho][Wo][C] (bf16, or fp32 with
 * out_dtype CONV3X3_DT_F32), channels fastest, both 16-byte aligned device
 * memory owned by the caller; f is a HOST array of kh*kw fp32 taps, row-major
 * [kh][kw], read during the call (the call copies it into the launch).
 * Arithmetic: fp32 accumulation, one rounding to bf16 on store.
 *
 * Limits: C a multiple of 8; 1 <= up, down <= UPFIRDN2D_MAX_FACTOR;
 * 1 <= kh, kw <= UPFIRDN2D_MAX_TAPS; 0 <= pads <= UPFIRDN2D_MAX_PAD (zeros only,
 * no cropping); Ho, Wo >= 1 and <= 65535; Wo * C / 8 < 2^31; N <= 65535.
 * Errors (conv3x3_status, see conv3x3.h): CONV3X3_ERR_INVALID_ARG for bad
 * sizes, factors, pads, pointers or dtype; CONV3X3_ERR_UNSUPPORTED beyond the
 * last two limits; CONV3X3_ERR_CUDA when the launch fails.
 * Asynchronous on `stream` (a cudaStream_t as void*); allocates nothing.
 */
#ifndef UPFIRDN2D_H
#define UPFIRDN2D_H

#ifdef __cplusplus
extern "C" {
#endif

#define UPFIRDN2D_MAX_TAPS 8
#define UPFIRDN2D_MAX_FACTOR 8
#define UPFIRDN2D_MAX_PAD 64

int upfirdn2d(const void* x, const float* f, void* y, int N, int C, int H, int W,
              int up, int down, int pad_x0, int pad_x1, int pad_y0, int pad_y1,
              int kh, int kw, int out_dtype, void* stream);

/* Output length along one axis (Ho from H, pad_y0, pad_y1, kh; Wo likewise),
 * or 0 when the arguments are outside the limits above.  Host only. */
int upfirdn2d_out_size(int len, int up, int down, int pad0, int pad1, int k);

#ifdef __cplusplus
}
#endif

#endif /* UPFIRDN2D_H */
