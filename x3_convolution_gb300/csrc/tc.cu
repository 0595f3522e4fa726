// tc.cu -- tensor-core (tcgen05 + TMEM + TMA) implicit-GEMM kernels for the
// pad-1 3x3 convolution on sm_103a (stride 1, and stride 2 for downsampling).
//
// Forward and dgrad share one persistent, warp-specialised kernel:
//   GEMM  M = N*H*W output pixels, N = output channels, K = 9 taps x channels.
//   A tile (128 pixels x 64 channels, one tap) arrives through a TMA im2col
//   tensor map: the hardware walks 128 consecutive output pixels, offsets each
//   by the tap, and zero-fills the halo -- no im2col buffer ever exists.
//   B tile comes from the KRSC weights with a tiled TMA map: K-major for the
//   forward (w[k][tap][c] is already [N][K]), MN-major for dgrad (w[k][tap][c]
//   read as [K=k][N=c]), so neither pass transposes anything in memory.  dgrad
//   mirrors the taps: dx = sum over (ra, sa) of dy at offset (ra-1, sa-1) times
//   w[:, 2-ra, 2-sa, :].
//   Warps 0-3 issue TMA, warp 4 owns TMEM and issues tcgen05.mma (128 x BN x 16,
//   fp32 accumulate), warps 5-12 drain the double-buffered TMEM accumulator:
//   bias + SiLU in fp32, round to bf16 (or keep fp32), store.  The 256-pixel x
//   128-channel tile can run transposed (weights as the M operand, both pixel
//   boxes as one N = 256 operand), and 256-channel tiles can run on two-CTA
//   clusters (k_igemm_pair: tcgen05 cta_group::2, M = 256 pixels per pair).
//
// Weight gradient: split-K implicit GEMM  M = Cout, N = (tap, Cin), K = pixels.
//   A = dy tile (64 pixels x 128 output channels, MN-major), B = im2col(x) for
//   three taps (64 pixels x 128 channels each, MN-major).  Each CTA owns one
//   (Cout block, tap row, Cin block) tile and one contiguous pixel range and
//   writes its fp32 partial tile to the caller's workspace; a second kernel
//   adds the partials in split order (deterministic).  dbias rides along: in
//   the CTAs that own it, the third tap's MMA is widened from N = 128 to 144
//   and its extra 16 columns read an 8 KB block of bf16 ones that sits right
//   after that tap's x tile in every stage (a separate N = 16 MMA costs about
//   as much as an N = 64 one).
//
// The subject page's kernels minimise memory transfers and avoid global
// transposes (clu0 C++/CUDA UNet diffusion, sourcepulse.org project page,
// "How It Works"); on sm_103a that is TMA im2col plus operand-major choices.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "act.cuh"
#include "conv3x3_internal.h"
#include "ptx.cuh"

namespace c3 {

int launch_wgrad_reduce2(const float* part, float* dw, float* db, long long dwsize, int Cout, int Sreg,
                         int S1, int S2, int k1, cudaStream_t st);
int launch_wgrad_reduce(const float* part, float* dw, float* db, long long dwsize, int Cout, int S,
                        int Sdb, cudaStream_t st);

namespace {

constexpr int BM = 128;              // output pixels per tile (MMA M, TMEM lanes)
constexpr int BKC = 64;              // channels per k-block: one 128-byte swizzle row
// Warp roles.  TMA copies issued by one thread do not overlap each other, so
// every stage's boxes are spread over kProd producer warps (warps 0..3); warp
// kProd allocates TMEM and issues the MMAs; the rest drain the accumulators.
constexpr int kProd = 4;
// How the producers share the im2col kernel's stages: each stage's boxes
// spread over all producers, or whole stages handed out round-robin.  The
// forward weight tile is one BN-row box or BN/64 boxes of 64 rows.
#ifndef C3_STAGE_PARALLEL
#define C3_STAGE_PARALLEL 1
#endif
#ifndef C3_ONE_WEIGHT_BOX
#define C3_ONE_WEIGHT_BOX 1
#endif

// SiLU in the forward epilogues through tanh (one special-function op) when
// 1, as z / (1 + e^-z) when 0
#ifndef C3_SILU_TANH
#define C3_SILU_TANH 1
#endif
constexpr bool kStageParallel = C3_STAGE_PARALLEL != 0;
constexpr bool kOneWeightBox = C3_ONE_WEIGHT_BOX != 0;
constexpr bool kWgStageParallel = false;  // the 3-stage wgrad ring is shared box-parallel
constexpr int kMmaWarp = kProd;
constexpr int kEpiBase = kProd + 1;
constexpr int kEpiWarps = 8;         // igemm: two epilogue warps per TMEM lane quarter
constexpr int kIgemmThreads = 32 * (kProd + 1 + kEpiWarps);
// block size of k_igemm: the transposed tile with the fused extras runs
// 2 + 1 + 12 warps
constexpr int igemm_threads(bool wide_epilogue) { return wide_epilogue ? 32 * 15 : kIgemmThreads; }
constexpr int kWgEpiWarps = 4;       // wgrad: one epilogue warp per lane quarter
constexpr int kThreads = 32 * (kProd + 1 + kWgEpiWarps);
constexpr uint32_t kABytes = BM * BKC * 2;
constexpr int kPlanSms = 152;        // split plan constant (shape-only workspace size)
constexpr size_t kGuardBytes = 16 * 1024;

// After an abort, copies still in flight land within microseconds; a stage
// whose other producers never issued their boxes will not complete, so the
// drain waits are kept short.
__device__ __forceinline__ unsigned long long drain_wait_ns(unsigned long long w) {
  return w < 50000000ULL ? w : 50000000ULL;
}

constexpr int pow2_cols(int n) { return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 512; }

// MT = pixel sub-tiles of 128 per CTA tile (two MMAs share each B stage when
// MT = 2, halving the B bytes per unit of tensor work).  KC = 64-channel chunks
// per stage: KC = 2 doubles the tensor work per pipeline round trip, which the
// single issuing thread needs when each chunk holds only 4 x N = 128 MMAs.
// Stage layout: KC chunks of A (MT boxes each), then KC chunks of B.
template <int BN, int MT, int KC = 1>
struct IgemmCfg {
  static constexpr uint32_t kChunkA = MT * kABytes;
  static constexpr uint32_t kChunkB = BN * BKC * 2;
  static constexpr uint32_t kATileBytes = KC * kChunkA;
  static constexpr uint32_t kBBytes = KC * kChunkB;
  static constexpr uint32_t kStageBytes = kATileBytes + kBBytes;
  static constexpr int kStages = (200 * 1024) / kStageBytes > 8 ? 8 : (200 * 1024) / kStageBytes;
  // producers take whole stages in turn when the ring is deep enough for that
  // (a parity wait is unambiguous only while S >= kProd); otherwise they split
  // each stage's boxes
  static constexpr bool kStagePar = kStageParallel && kStages >= kProd;
  static constexpr int kTmemCols = pow2_cols(2 * MT * BN);
  static_assert(2 * MT * BN <= 512, "double-buffered accumulators must fit in TMEM");
  // epilogue warps' bias slices (after the barriers): kEpiCols columns each
  static constexpr int kEpiCols = MT == 2 ? BN : BN / 2;
  static constexpr uint32_t kBiasBytes = (uint32_t)kEpiWarps * kEpiCols * 4;
  // + barriers, + bias slices, + alignment slack, + a 16 KB guard so that no
  // descriptor arithmetic can ever address past the allocation
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + 256 + kBiasBytes + 1024 + kGuardBytes;
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

struct IgemmParams {
  void* out;
  const float* bias;
  int act, out_f32;
  int P, H, W;
  int kchunks;    // ceil(A channels / 64)
  int kgroups;    // k-blocks per tap: ceil(kchunks / KC)
  // Pixel traversal: P pixels of an (N, H, W) grid -- the output grid of the
  // forward, dx's grid of a stride-1 dgrad, dy's grid of a stride-2 dgrad.
  int ustride;    // forward: input row/column step per output pixel (1 or 2)
  int s2;         // dgrad of a stride-2 conv, run as four output-parity classes
  int oh, ow;     // s2: dx's H and W
  int kchunks_a;  // forward, channel-split input: chunks [0, kchunks_a) come from tmA, the rest from tmA2
  int nout;       // output channels (Cout fwd, Cin dgrad)
  int nsplit;     // output columns [0, nsplit) go to out (row stride nsplit), [nsplit, nout) to out2
  int num_m_tiles, num_n_tiles;
  unsigned* status;
  unsigned long long wait_ns;
  void* out2 = nullptr;
  // forward: also store z = conv + bias, rounded once to bf16, laid out like out
  __nv_bfloat16* zout = nullptr;
  // dgrad: scale by act'(zin) (the input's pre-activation, split like the output)
  const __nv_bfloat16* zin = nullptr;
  const __nv_bfloat16* zin2 = nullptr;
  int zin_act = CONV3X3_ACT_NONE;
  // bf16 output through TMA stores of {64 channels, 32 pixels} boxes (map
  // tmY), staged in the idle stage ring: set only where every CTA (or pair)
  // has one tile and the output is one plain bf16 tensor
  int epi_tma = 0;
  // 256-channel pair tiles: work items from half_from on are half-width tiles
  // of 128 channels, two per remaining tile (the last round's tiles split so
  // that they spread over the pairs instead of leaving most of them idle)
  int half_from = 0x7fffffff;
};

// Where output column col0 of pixel `pix` lives.  Columns [0, nsplit) are in
// the primary tensor (row stride nsplit); columns [nsplit, nout) -- the second
// part of a channel-split input gradient -- in the second one (row stride
// nout - nsplit).  nsplit is a multiple of 32, so a 32-column chunk never
// straddles the two.  `lim` = columns left in that tensor's row from col0.
struct OutPos {
  long long off;
  int lim;
  bool second;
};

__device__ __forceinline__ OutPos out_pos(const IgemmParams& p, long long pix, int col0) {
  if (col0 < p.nsplit) return OutPos{pix * p.nsplit + col0, p.nsplit - col0, false};
  return OutPos{pix * (p.nout - p.nsplit) + (col0 - p.nsplit), p.nout - col0, true};
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* o, int lim, const float (&f)[32]) {
#pragma unroll
  for (int g = 0; g < 4; ++g)
    if (8 * g < lim) {
      uint4 u;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[8 * g + 2 * i], f[8 * g + 2 * i + 1]);
      *reinterpret_cast<uint4*>(o + 8 * g) = u;
    }
}

// The 32 z_in values (bf16) of one output chunk, fetched before the
// accumulator so that their latency overlaps the TMEM load.
__device__ __forceinline__ void load_zin(const IgemmParams& p, long long pix, int col0,
                                         uint4 (&zr)[4]) {
  const OutPos o = out_pos(p, pix, col0);
  const __nv_bfloat16* zp = (o.second ? p.zin2 : p.zin) + o.off;
#pragma unroll
  for (int g = 0; g < 4; ++g)
    zr[g] = 8 * g < o.lim ? __ldg(reinterpret_cast<const uint4*>(zp + 8 * g))
                          : make_uint4(0u, 0u, 0u, 0u);
}

// L2 prefetch of one output row's z_in over columns [col0, col0 + ncols),
// issued while the tile's MMAs still run: one prefetch at the start of each
// 32-column chunk (an address that chunk itself reads).
__device__ __forceinline__ void prefetch_zin_row(const IgemmParams& p, long long pix, int col0,
                                                 int ncols) {
  const int end = min(col0 + ncols, p.nout);
  for (int c = col0; c < end; c += 32) {
    const OutPos o = out_pos(p, pix, c);
    asm volatile("prefetch.global.L2 [%0];" ::"l"((o.second ? p.zin2 : p.zin) + o.off));
  }
}

// The 32 bias values of one output chunk (zero past nout), loaded ahead of the
// accumulator: with the loads issued before the TMEM load, the bias add does
// not wait on them.
__device__ __forceinline__ void load_bias(const IgemmParams& p, int col0, float (&bv)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const float4 b = col0 + i < p.nout ? __ldg(reinterpret_cast<const float4*>(p.bias + col0 + i))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
    bv[i] = b.x;
    bv[i + 1] = b.y;
    bv[i + 2] = b.z;
    bv[i + 3] = b.w;
  }
}

// The bias of one epilogue warp's kCols output columns c0 .. c0 + kCols - 1
// (zero at or past nout), staged in the warp's own shared-memory slice before
// it waits for the accumulator.  A tile's chunks then read it from shared
// memory instead of each waiting on a global load: with one tile per CTA (the
// 8x8 and 16x16 layers) nothing else hides that latency.
template <int kCols>
__device__ __forceinline__ void stage_bias_slice(const IgemmParams& p, int c0, float* sl, int lane) {
  __syncwarp();  // every lane is done with the previous tile's slice
#pragma unroll
  for (int i = lane; i < kCols; i += 32) sl[i] = c0 + i < p.nout ? __ldg(p.bias + c0 + i) : 0.0f;
  __syncwarp();
}

__device__ __forceinline__ void bias_from_slice(const float* sl, float (&bv)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const float4 b = *reinterpret_cast<const float4*>(sl + i);  // one address for the warp
    bv[i] = b.x;
    bv[i + 1] = b.y;
    bv[i + 2] = b.z;
    bv[i + 3] = b.w;
  }
}

// Activation (kAct), then the fused z_in scaling (act'(z_in)), on one chunk
// in fp32.
template <bool kExt, bool kTanh, bool kAct = true>
__device__ __forceinline__ void epi_act_zin(const IgemmParams& p, float (&f)[32], const uint4 (&zr)[4]) {
  if (kAct && p.act == CONV3X3_ACT_SILU) {
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = kTanh ? silu_tanh_f32(f[i]) : silu_f32(f[i]);
  } else if (kAct && p.act == CONV3X3_ACT_LRELU) {
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = f[i] >= 0.0f ? f[i] : 0.2f * f[i];
  }
  if (kExt && p.zin) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&zr[g]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 z = __bfloat1622float2(h[i]);
        f[8 * g + 2 * i] *= act_grad_f32(p.zin_act, z.x);
        f[8 * g + 2 * i + 1] *= act_grad_f32(p.zin_act, z.y);
      }
    }
  }
}

// One 32-column chunk of the TMA-store epilogue (epi_tma): bias, activation
// and z_in scaling in fp32 as in store_chunk, one bf16 rounding, and the
// thread's 64 bytes staged as 16-byte pieces c0 .. c0 + 3 of its 128-byte row
// `row` of a {64 channels, 32 pixels} box, piece c at c ^ (lane % 8) (the
// 128-byte swizzle: eight rows of a store phase cover all 32 banks).  kPass
// as in store_chunk.
template <bool kExt, int kPass = 2, bool kTanh = C3_SILU_TANH>
__device__ __forceinline__ void stage_chunk_bf16(const IgemmParams& p, const uint32_t (&v)[32],
                                                 const float (&bv)[32], const uint4 (&zr)[4], uint8_t* row,
                                                 int c0, int lane) {
  constexpr bool kFwd = kPass != 1, kDg = kPass != 0;
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]) + ((kFwd && p.bias) ? bv[i] : 0.0f);
  epi_act_zin<kExt && kDg, kTanh, kFwd>(p, f, zr);
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[8 * g + 2 * i], f[8 * g + 2 * i + 1]);
    *reinterpret_cast<uint4*>(row + (((c0 + g) ^ (lane & 7)) << 4)) = u;
  }
}

// Epilogue of one 32-column chunk: (+ bias) -> [store z] -> activation ->
// [* act'(z_in)] -> fp32 or bf16 store.  kExt = false compiles out the fused
// extras (z store, z_in scaling, split output) for the plain calls.  kPass
// tells the pass at compile time -- 0 forward (bias, z store, activation),
// 1 input gradient (z_in scaling, split output), 2 either, from the run-time
// fields -- so that a fused tile keeps only its own pass's operands live.
// kTanh takes SiLU through tanh (silu_tanh_f32).
template <bool kExt, int kPass = 2, bool kTanh = C3_SILU_TANH>
__device__ __forceinline__ void store_chunk(const IgemmParams& p, long long pix, int col0,
                                            const uint32_t (&v)[32], const float (&bv)[32],
                                            const uint4 (&zr)[4]) {
  constexpr bool kFwd = kPass != 1, kDg = kPass != 0;
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
  if (kFwd && p.bias) {
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] += bv[i];
  }
  if (kExt && kFwd && p.zout) store_bf16x32(p.zout + pix * p.nout + col0, p.nout - col0, f);
  epi_act_zin<kExt && kDg, kTanh, kFwd>(p, f, zr);
  const OutPos o = (kExt && kDg) ? out_pos(p, pix, col0) : OutPos{pix * p.nout + col0, p.nout - col0, false};
  void* base = (kExt && kDg && o.second) ? p.out2 : p.out;
  if (p.out_f32) {
    float* op = static_cast<float*>(base) + o.off;
#pragma unroll
    for (int g = 0; g < 4; ++g)
      if (8 * g < o.lim) {
        reinterpret_cast<float4*>(op + 8 * g)[0] = make_float4(f[8 * g], f[8 * g + 1], f[8 * g + 2], f[8 * g + 3]);
        reinterpret_cast<float4*>(op + 8 * g)[1] = make_float4(f[8 * g + 4], f[8 * g + 5], f[8 * g + 6], f[8 * g + 7]);
      }
  } else {
    store_bf16x32(static_cast<__nv_bfloat16*>(base) + o.off, o.lim, f);
  }
}

// All features, operands fetched here (the halo and 8-channel kernels).
__device__ __forceinline__ void store_chunk(const IgemmParams& p, long long pix, int col0,
                                            const uint32_t (&v)[32]) {
  float bv[32];
  if (p.bias) load_bias(p, col0, bv);
  uint4 zr[4] = {};
  if (p.zin) load_zin(p, pix, col0, zr);
  store_chunk<true>(p, pix, col0, v, bv, zr);
}

// ----------------------------------------------------------------------------
// forward / dgrad implicit GEMM
// ----------------------------------------------------------------------------
// Stride-2 dgrad by output parity.  dx[h][w] collects dy[ho][wo] w[r][s] over
// 2 ho + r - 1 = h, 2 wo + s - 1 = w.  For h = 2i + ph only rows r = ph + 1
// (mod 2) contribute, from dy row i + (ph + 1 - r) / 2: one tap row (r = 1)
// for even h, two (r = 0 -> i + 1, r = 2 -> i) for odd h; columns likewise.
// Each class (ph, pw) is a stride-1 implicit GEMM over dy's pixel grid with
// 1, 2, 2 or 4 taps, all of them reading a 2x2 window at (i, j): the nine
// taps are each used once, as in the stride-1 dgrad.
struct TileInfo {
  int mt, nt, cls, kblocks;
};

__device__ __forceinline__ int igemm_num_tiles(const IgemmParams& p, bool s2) {
  return (s2 ? 4 : 1) * p.num_m_tiles * p.num_n_tiles;
}

__device__ __forceinline__ TileInfo tile_info(const IgemmParams& p, int tile, bool s2) {
  if (!s2) return TileInfo{tile / p.num_n_tiles, tile % p.num_n_tiles, 0, 9 * p.kgroups};
  const int per = p.num_m_tiles * p.num_n_tiles;
  const int ci = tile / per, rest = tile - ci * per;
  const int cls = 3 - ci;  // cls = 2 ph + pw; the 4-tap class first
  const int ntaps = (1 + (cls >> 1)) * (1 + (cls & 1));
  return TileInfo{rest / p.num_n_tiles, rest % p.num_n_tiles, cls, ntaps * p.kgroups};
}

// Tap `t` of class `cls`: weight tap r*3+s and the A window offsets (dj, di).
__device__ __forceinline__ void s2_tap(int cls, int t, int& wtap, int& dj, int& di) {
  const int ph = cls >> 1, pw = cls & 1, ns = 1 + pw;
  const int ri = t / ns, si = t - ri * ns;
  const int r = ph ? 2 * ri : 1, s = pw ? 2 * si : 1;
  wtap = r * 3 + s;
  di = (ph + 1 - r) >> 1;
  dj = (pw + 1 - s) >> 1;
}
// kExt = false: no fused extras and no stride-2 dgrad (p.s2, p.zout, p.zin
// and the split output are ignored).
//
// kT (128-channel x 256-pixel tiles only): the transposed product.  The weight
// tile is the MMA's A operand (M = 128 output channels) and the two im2col
// boxes, contiguous in the stage, are one N = 256 B operand, so each K step
// is one 128 x 256 x 16 MMA instead of two 128 x 128 x 16 ones sharing B:
// the same tensor work with a third fewer operand bytes read from shared
// memory per MMA and half the instructions for the issuing thread.  The
// accumulator then holds channels on TMEM lanes and pixels on columns, and
// the epilogue stores one channel per thread (and, for a fused dgrad, loads
// that channel's z_in the same way).  No stride-2 dgrad (the dispatch sends
// it to the untransposed tile).
template <int BN, int MT, bool kDgrad, bool kExt, int KC, bool kT = false>
__global__ void __launch_bounds__(igemm_threads(kT && kExt), 1)
    k_igemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
            const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmY,
            const IgemmParams p) {
  static_assert(!kT || (MT == 2 && BN == BM && KC == 1), "transposed tiles are 128 channels x 256 pixels");
  using Cfg = IgemmCfg<BN, MT, KC>;
  constexpr int S = Cfg::kStages;
  constexpr int TM = BM * MT;  // pixels per CTA tile
  // Warp roles: NP TMA producer warps, the MMA warp, NE epilogue warps.  The
  // transposed tile with the fused extras, whose epilogue (one channel per
  // thread, z loads or stores per element) outlasts its main loop, runs two
  // producer warps and twelve epilogue warps (three per TMEM lane quarter):
  // 128-channel 64x64 fused dgrad 88 -> 74 us.  The plain transposed tile
  // keeps four producers and eight epilogue warps: with one producer its main
  // loop, which sets its pace, ran 2.5 us longer.
  constexpr bool kWide = kT && kExt;
  constexpr int NP = kWide ? 2 : kProd, MW = NP, EB = NP + 1, NE = kWide ? 12 : kEpiWarps;
  static_assert(32 * (NP + 1 + NE) == igemm_threads(kWide), "warp roles and block size");
  // A producer's parity wait on a stage is unambiguous only while no producer
  // can run a whole ring ahead: stage-parallel mode needs S >= NP.
  constexpr bool kSP = kWide ? kStageParallel && S >= NP : Cfg::kStagePar;
  static_assert(!kSP || S >= NP, "stage-parallel producers need S >= NP");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * Cfg::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  const bool s2 = kExt && kDgrad && !kT && p.s2;  // stride-2 dgrad by output parity
  const int num_tiles = igemm_num_tiles(p, s2);
  const int HW = p.H * p.W;

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], kSP ? 1 : NP);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], NE);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    if (p.kchunks_a < p.kchunks) tma_prefetch_desc(&tmA2);
    tma_prefetch_desc(&tmB);
  }
  if (warp == MW) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel's writes are visible from here on

  if (warp < NP) {
    // ------------------------------------------------------------ TMA producers
    // Stage boxes: MT im2col A boxes (128 pixels x 64 channels) then BN/64
    // weight boxes (64 rows x 64 channels); producer `warp` issues box b when
    // b % NP == warp and registers its own byte count on the full barrier.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const TileInfo ti = tile_info(p, tile, s2);
        const int mt = ti.mt, nt = ti.nt;
        // window origin of each 128-pixel sub-tile: the input pixel (u*h - 1,
        // u*w - 1) of the first output pixel (stride u, pad 1), or dy's pixel
        // itself for the parity classes of a stride-2 dgrad
        int cw[MT], ch[MT], cn[MT];
#pragma unroll
        for (int u = 0; u < MT; ++u) {
          const int p0 = mt * TM + u * BM;
          const int n0 = p0 / HW, rem = p0 - n0 * HW;
          const int h0 = rem / p.W;
          cn[u] = n0;
          ch[u] = s2 ? h0 : p.ustride * h0 - 1;
          cw[u] = s2 ? rem - h0 * p.W : p.ustride * (rem - h0 * p.W) - 1;
        }
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          const int tap = kb / p.kgroups, cg = (kb - tap * p.kgroups) * KC;
          // A window offsets and weight tap of this k-block
          int wtap, off_w, off_h;
          if (s2) {
            s2_tap(ti.cls, tap, wtap, off_w, off_h);
          } else {
            off_w = tap % 3;
            off_h = tap / 3;
            wtap = kDgrad ? 8 - tap : tap;
          }
          // stage-parallel mode: this producer owns every NP-th stage
          const bool mine = kSP ? (issued % NP == warp) : true;
          if (mine) {
            if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns, p.status, abort_flag)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + (size_t)stage * Cfg::kStageBytes;
            uint8_t* sb = sa + Cfg::kATileBytes;
            // boxes: MT im2col A boxes, then the weight tile as one BN-row box
            // (forward, K-major) or BN/64 boxes of 64 rows
            constexpr bool kOneB = !kDgrad && kOneWeightBox;
            constexpr int kBBoxes = kOneB ? 1 : BN / 64;
            constexpr uint32_t kBBox = kOneB ? (uint32_t)BN * 128u : 8192u;
            constexpr int kPer = MT + kBBoxes;  // boxes per chunk
            constexpr int kBoxes = KC * kPer;
            uint32_t bytes = 0;
#pragma unroll
            for (int b = 0; b < kBoxes; ++b)
              if (kSP || b % NP == warp) bytes += b % kPer < MT ? kABytes : kBBox;
            mbar_arrive_expect_tx(&full[stage], bytes);
#pragma unroll
            for (int b = 0; b < kBoxes; ++b) {
              if (!kSP && b % NP != warp) continue;
              // chunk cc of the stage (a chunk past the channels reads zeros)
              const int c = b / kPer, r = b - c * kPer, cc = cg + c;
              if (r < MT) {
                // channel-split input: chunks past kchunks_a read the second tensor
                const bool second = cc >= p.kchunks_a;
                tma_load_im2col_4d(sa + c * Cfg::kChunkA + r * kABytes, second ? &tmA2 : &tmA,
                                   &full[stage], (second ? cc - p.kchunks_a : cc) * BKC, cw[r],
                                   ch[r], cn[r], (uint16_t)off_w, (uint16_t)off_h);
              } else {
                const int j = r - MT;
                uint8_t* dst = sb + c * Cfg::kChunkB;
                if (!kDgrad)
                  tma_load_3d(dst + j * kBBox, &tmB, &full[stage], cc * BKC, wtap, nt * BN + j * 64);
                else
                  tma_load_3d(dst + j * 8192, &tmB, &full[stage], nt * BN + j * 64, wtap, cc * BKC);
              }
            }
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // drain: wait (bounded) for every load still in flight before exiting
        int n = issued < S ? issued : S;
        int st = stage;
        uint32_t ph = phase;
        for (int i = 0; i < n; ++i) {
          if (--st < 0) {
            st = S - 1;
            ph ^= 1;
          }
          mbar_wait(&full[st], ph, drain_wait_ns(p.wait_ns), nullptr, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == MW) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0, kDgrad ? 1 : 0);
      // transposed: the weight tile (K-major forward, MN-major dgrad) is A
      constexpr uint32_t idesc_t = idesc_bf16_f32(BM, MT * BM, kDgrad ? 1 : 0, 0);
      // One thread issues every MMA, and its instruction path per k-block
      // sets the pace when the MMAs are short (N = 128: 64 cycles each), so
      // the descriptors are built once: a stage, a sub-tile or a K step only
      // moves the start-address field (bits 0-13, 16-byte units), and no
      // offset inside the shared-memory allocation carries out of it.
      const uint32_t sbase = smem_u32(smem);
      const uint64_t a_desc0 = smem_desc(sbase, 16, 1024, kSwizzle128B);
      const uint64_t b_desc0 = kDgrad ? smem_desc(sbase + Cfg::kATileBytes, 8192, 1024, kSwizzle128B)
                                      : smem_desc(sbase + Cfg::kATileBytes, 16, 1024, kSwizzle128B);
      constexpr uint32_t kStageStep = Cfg::kStageBytes >> 4;
      constexpr uint32_t kBKStep = (kDgrad ? 2048u : 32u) >> 4;  // per K step of 16
      constexpr uint32_t kAKStep = 32u >> 4;
      constexpr uint32_t kSubStep = kABytes >> 4;
      int stage = 0;
      uint32_t phase = 0, stage_off = 0;
      int buf = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        if (!mbar_wait(&tempty[buf], acc_phase ^ 1, p.wait_ns, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * MT * BN);
        const int kblocks = tile_info(p, tile, s2).kblocks;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.wait_ns, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a_desc0 + stage_off, bd = b_desc0 + stage_off;
          const uint32_t acc0 = kb != 0 ? 1u : 0u;  // the tile's first K step starts the sum
          if constexpr (kT) {
            // weights (M = 128 channels) x both pixel boxes (N = 256)
#pragma unroll
            for (int k = 0; k < BKC / 16; ++k)
              tc_mma_bf16(d_tmem, bd + (uint64_t)(k * kBKStep), ad + (uint64_t)(k * kAKStep), idesc_t,
                          k == 0 ? acc0 : 1u);
          } else {
#pragma unroll
            for (int c = 0; c < KC; ++c)
#pragma unroll
              for (int k = 0; k < BKC / 16; ++k)
#pragma unroll
                for (int u = 0; u < MT; ++u)
                  tc_mma_bf16(d_tmem + (uint32_t)(u * BN),
                              ad + (uint64_t)(c * (Cfg::kChunkA >> 4) + u * kSubStep + k * kAKStep),
                              bd + (uint64_t)(c * (Cfg::kChunkB >> 4) + k * kBKStep), idesc,
                              (c == 0 && k == 0) ? acc0 : 1u);
          }
          tc_commit(&empty[stage]);
          stage_off += kStageStep;
          if (++stage == S) {
            stage = 0;
            stage_off = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[buf]);
        if (++buf == 2) {
          buf = 0;
          acc_phase ^= 1;
        }
      }
      // make sure every issued MMA has retired before TMEM is released
      tc_commit(drain);
      mbar_wait(drain, 0, p.wait_ns, nullptr, nullptr);
    }
    __syncwarp();
  } else if constexpr (kT) {
    // ------------------------------------------------------------ epilogue (transposed)
    // TMEM lane = output channel, column = pixel of the 256-pixel tile.  Warp
    // w reads lanes 32*(w%4) .. +31 (32 channels); the NE / 4 warps of a lane
    // quarter take the tile's eight 32-pixel chunks in turn (part, part +
    // NE / 4, ...).  A thread owns one channel, so a chunk leaves as 32 scalar stores,
    // each a 64-byte (bf16) or 128-byte (fp32) contiguous run across the warp.
    constexpr int kParts = NE / 4, kChunks = TM / 32;
    const int q = warp & 3;
    const int part = (warp - EB) >> 2;
    int buf = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const TileInfo ti = tile_info(p, tile, false);
      const int ch = ti.nt * BN + q * 32 + lane;
      const bool ch_ok = ch < p.nout;
      const float bc = (p.bias && ch_ok) ? __ldg(p.bias + ch) : 0.0f;
      // this channel's tensor, row stride and column (the split output of a
      // channel-split dgrad puts channels [nsplit, nout) in the second tensor)
      const bool second = kExt && ch >= p.nsplit;
      void* obase = second ? p.out2 : p.out;
      const long long ostride = !kExt ? p.nout : second ? p.nout - p.nsplit : p.nsplit;
      const int ocol = second ? ch - p.nsplit : ch;
      const long long pix_base = (long long)ti.mt * TM;
      if (kExt && p.zin && ch_ok) {
        // L2 prefetch of the z_in the warp reads for this tile (its 32
        // channels, one 64-byte run per pixel) while the MMAs still run
        const __nv_bfloat16* zq = (second ? p.zin2 : p.zin) + (ocol - lane);
#pragma unroll 1
        for (int k = part; k < kChunks; k += kParts) {
          const long long px = pix_base + k * 32 + lane;
          if (px < p.P) asm volatile("prefetch.global.L2 [%0];" ::"l"(zq + px * ostride));
        }
      }
      if (!mbar_wait(&tfull[buf], acc_phase, p.wait_ns, p.status, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * MT * BN);
#pragma unroll 1
      for (int j = part; j < kChunks; j += kParts) {
        const long long pix0 = pix_base + j * 32;
        const int npix = p.P - pix0 < 32 ? (int)(p.P - pix0) : 32;  // <= 0 past the end
        // z_in of this channel at the chunk's 32 pixels (fused dgrad), loaded
        // ahead of the accumulator: a warp's load reads 32 adjacent channels
        // of one pixel, one 64-byte run, as its stores below write
        unsigned short zr[32];
        if (kExt && p.zin && ch_ok) {
          const unsigned short* zp =
              reinterpret_cast<const unsigned short*>(second ? p.zin2 : p.zin) + pix0 * ostride + ocol;
          // this warp's next chunk's 32 pixels into L1 (one 64-byte run per
          // lane) while this chunk is processed; this chunk's were fetched
          // during the previous one (or, for the first, come from L2)
          if (j + kParts < kChunks && pix0 + 32 * kParts + lane < p.P)
            asm volatile("prefetch.global.L1 [%0];" ::"l"(zp - lane + (32 * kParts + lane) * ostride));
#pragma unroll
          for (int i = 0; i < 32; ++i) zr[i] = i < npix ? __ldg(zp + i * ostride) : (unsigned short)0;
        }
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + (uint32_t)(j * 32), v);
        tmem_ld_wait();
        if (ch_ok && npix > 0) {
          float f[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]) + bc;
          if (kExt && p.zout) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < npix) p.zout[(pix0 + i) * p.nout + ch] = __float2bfloat16_rn(f[i]);
          }
          if (p.act == CONV3X3_ACT_SILU) {
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = C3_SILU_TANH ? silu_tanh_f32(f[i]) : silu_f32(f[i]);
          } else if (p.act == CONV3X3_ACT_LRELU) {
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = f[i] >= 0.0f ? f[i] : 0.2f * f[i];
          }
          if (kExt && p.zin) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              f[i] *= act_grad_f32(p.zin_act, __bfloat162float(__ushort_as_bfloat16(zr[i])));
          }
          if (p.out_f32) {
            float* op = static_cast<float*>(obase) + pix0 * ostride + ocol;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < npix) op[i * ostride] = f[i];
          } else {
            __nv_bfloat16* op = static_cast<__nv_bfloat16*>(obase) + pix0 * ostride + ocol;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < npix) op[i * ostride] = __float2bfloat16_rn(f[i]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      if (++buf == 2) {
        buf = 0;
        acc_phase ^= 1;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warp w may read TMEM lanes 32*(w%4) .. +31.  The two warps of a lane
    // quarter take one 128-pixel sub-tile each (MT = 2) or half the columns
    // of the single sub-tile (MT = 1).
    constexpr int kCols = Cfg::kEpiCols;
    const int q = warp & 3;
    const int half = (warp - EB) >> 2;
    const int sub = MT == 2 ? half : 0;
    const int col_off = MT == 2 ? 0 : half * kCols;
    const int row = q * 32 + lane;
    float* bsl = reinterpret_cast<float*>(smem + (size_t)S * Cfg::kStageBytes + 256) + (warp - EB) * kCols;
    int buf = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const TileInfo ti = tile_info(p, tile, s2);
      const int mt = ti.mt, nt = ti.nt;
      long long pix = (long long)mt * TM + sub * BM + row;
      bool valid = pix < p.P;
      if (s2 && valid) {
        // dy pixel (n, i, j) of class (ph, pw) -> dx pixel (n, 2i + ph, 2j + pw)
        const int n = (int)(pix / HW), rem = (int)(pix - (long long)n * HW);
        const int i = rem / p.W, j = rem - i * p.W;
        const int h = 2 * i + (ti.cls >> 1), w = 2 * j + (ti.cls & 1);
        valid = h < p.oh && w < p.ow;
        pix = ((long long)n * p.oh + h) * p.ow + w;
      }
      if (kExt && kDgrad && p.zin && valid && nt * BN + col_off < p.nout)
        prefetch_zin_row(p, pix, nt * BN + col_off, kCols);
      if (!kDgrad && p.bias) stage_bias_slice<kCols>(p, nt * BN + col_off, bsl, lane);
      if (!mbar_wait(&tfull[buf], acc_phase, p.wait_ns, p.status, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) +
                             (uint32_t)((buf * MT + sub) * BN + col_off);
      // the TMA-store path serves every tile of one-tile CTAs (epi_tma 1) or
      // each CTA's last tile (epi_tma 2): there the stage ring is idle
      const bool tma_here = p.epi_tma == 1 || (p.epi_tma == 2 && tile + (int)gridDim.x >= num_tiles);
      if constexpr (kCols % 64 == 0) {
        if (tma_here) {
          // every MMA of the tile has completed, so no stage is in use; this
          // warp's 32 pixels leave as kCols / 64 boxes of {64 channels, 32 pixels}
          uint8_t* stg = smem + (size_t)(warp - EB) * (kCols / 64) * 4096u;
          const long long wrow0 = (long long)mt * TM + sub * BM + q * 32;
#pragma unroll 1
          for (int j = 0; j < kCols / 32; ++j) {
            const int col0 = nt * BN + col_off + j * 32;
            float bv[32];
            if (!kDgrad && p.bias) bias_from_slice(bsl + j * 32, bv);
            uint4 zr[4] = {};
            if (kExt && kDgrad && p.zin && valid && col0 < p.nout) load_zin(p, pix, col0, zr);
            uint32_t v[32];
            tmem_ld_32x32b_x32(taddr + (uint32_t)(j * 32), v);
            tmem_ld_wait();
            uint8_t* box = stg + (j >> 1) * 4096u;
            stage_chunk_bf16<kExt, kDgrad ? 1 : 0>(p, v, bv, zr, box + lane * 128, (j & 1) * 4, lane);
            if (j & 1) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0 && col0 - 32 < p.nout && wrow0 < p.P) tma_store_2d(&tmY, box, col0 - 32, (int)wrow0);
            }
          }
          if (lane == 0) {
            bulk_commit();
            bulk_wait_read<0>();  // the stores' writes complete with the grid
          }
          __syncwarp();
        }
      }
#pragma unroll 1
      for (int j = 0; j < (tma_here && kCols % 64 == 0 ? 0 : kCols / 32); ++j) {
        const int col0 = nt * BN + col_off + j * 32;
        const bool live = valid && col0 < p.nout;
        // operands that do not depend on the accumulator are loaded first
        float bv[32];
        if (!kDgrad && p.bias && live) bias_from_slice(bsl + j * 32, bv);
        uint4 zr[4] = {};
        if (kExt && kDgrad && p.zin && live) load_zin(p, pix, col0, zr);
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + (uint32_t)(j * 32), v);
        tmem_ld_wait();
        if (live) store_chunk<kExt, kDgrad ? 1 : 0>(p, pix, col0, v, bv, zr);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      if (++buf == 2) {
        buf = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == MW) tmem_dealloc(tmem_base, Cfg::kTmemCols);
}

// ----------------------------------------------------------------------------
// forward / dgrad implicit GEMM on CTA pairs (tcgen05 cta_group::2)
// ----------------------------------------------------------------------------
// A cluster of two CTAs on two SMs owns one tile of 256 pixels x 256 output
// channels.  Each CTA stages its own 128 pixels (one im2col A box) and half of
// the weight tile (128 of the 256 channels); one thread of rank 0 issues
// M = 256, N = 256 MMAs that read A and B from both CTAs' shared memory, and
// each CTA's TMEM accumulates its 128 pixels x 256 channels.  Per SM that is
// the tensor work of a 128 x 256 tile for two thirds of its operand bytes
// (32 KB per 64-channel k-block instead of 48), so six stages fit where four
// did and the ring covers 50 % more load and MMA latency.
//
// Barriers.  full[s] of rank 0 counts both CTAs' bytes (each CTA's loads
// signal it through the cluster window, rank 0's producer registers the
// pair's total); empty[s] and tfull[b] exist in both CTAs and are signalled by
// rank 0's multicast commits; tempty[b] of rank 0 collects the epilogue warps
// of both CTAs.  Every wait is bounded; the two cluster barriers (after setup,
// before the TMEM release) are reached by every thread on every path.
//
// The pair tile is 256 pixels x BN output channels, BN in {128, 192, 256}:
// each CTA stages BN / 2 weight rows (the forward's K-major box of BN / 2 rows;
// dgrad's MN-major boxes of 64 channels, the last one partly unused when
// BN / 2 = 96), the MMA is M = 256, N = BN.  KC = 64-channel chunks per stage:
// with KC = 2 a barrier round trip of the issuing thread covers eight MMAs
// (1024 cycles of tensor work at N = 256) instead of four; the three 64 KB
// stages are then filled box-parallel by all producers.
//
// BN = 384 (one accumulator, 384 of the 512 TMEM columns): an M = 256,
// N = 256 and an M = 256, N = 128 MMA per K step.  CTA r stages output
// channels [128 r, 128 r + 128) as its weight rows 0-127 and [256 + 64 r,
// 256 + 64 r + 64) as rows 128-191, so the first MMA (rows 0-127 of both CTAs)
// writes accumulator columns 0-255 and the second (rows 128-191) columns
// 256-383: column = channel of the tile.  Both passes load three 64-row (or
// 64-channel) boxes per CTA and k-block, every byte used.
// Work item `it` of a 256-channel pair launch: tiles [0, half_from) whole,
// then every remaining tile as two items of 128 channels each (N = 128 MMAs,
// 64 weight rows per CTA), channel offset 0 or 128 within the tile.
struct PairItem {
  int tile, coff;
  bool half;
};
__device__ __forceinline__ PairItem pair_item(const IgemmParams& p, int it) {
  if (it < p.half_from) return PairItem{it, 0, false};
  const int h = it - p.half_from;
  return PairItem{p.half_from + (h >> 1), (h & 1) * 128, true};
}
__device__ __forceinline__ int pair_num_items(const IgemmParams& p, int num_tiles) {
  return p.half_from < num_tiles ? 2 * num_tiles - p.half_from : num_tiles;
}

template <int BN, bool kDgrad, int KC = 1>
struct PairCfg {
  static constexpr int kHalf = BN / 2;                  // weight rows (output channels) per CTA
  static constexpr int kDgradBoxes = (kHalf + 63) / 64;  // dgrad: 64-channel MN-major boxes
  static constexpr uint32_t kBHalf = kDgrad ? (uint32_t)kDgradBoxes * 8192u : (uint32_t)kHalf * 128u;
  static constexpr int kBufs = 2 * BN <= 512 ? 2 : 1;    // TMEM accumulators
  static constexpr uint32_t kStage = KC * (kABytes + kBHalf);  // per CTA: KC A boxes, then KC B halves
  static constexpr int kStagesFit = (int)((200u * 1024u) / kStage);
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static constexpr bool kSP = kStages >= kProd;  // whole stages per producer, else boxes
  // epilogue warps' bias slices (after the barriers): BN / 2 columns each
  static constexpr uint32_t kBiasBytes = (uint32_t)kEpiWarps * kHalf * 4;
  static constexpr size_t kSmem = (size_t)kStages * kStage + 256 + kBiasBytes + 1024 + kGuardBytes;
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
  static_assert(BN == 128 || BN == 192 || BN == 256 || BN == 384, "pair tiles are 128 .. 384 channels wide");
  static_assert(BN != 384 || KC == 1, "384-channel pair tiles take one chunk per stage");
  static_assert(KC == 1 || KC == 2, "one or two chunks per stage");
  static_assert(kStage % 1024 == 0, "stages must keep 1 KB swizzle alignment");
  static_assert(kStages >= 2, "pair stage ring too shallow");
};

template <bool kDgrad, bool kExt, int BN = 256, int KC = 1>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kIgemmThreads, 1)
    k_igemm_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                 const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
                 const __grid_constant__ CUtensorMap tmY, const IgemmParams p) {
  using Cfg = PairCfg<BN, kDgrad, KC>;
  constexpr int S = Cfg::kStages;
  constexpr bool kSP = Cfg::kSP;
  constexpr int kPairBN = BN;
  constexpr uint32_t kPairStage = Cfg::kStage;
  extern __shared__ uint8_t smem_raw[];
  // same offset in both CTAs: the MMAs address the peer's operands at the
  // offsets of rank 0's
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * kPairStage);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
  const int num_tiles = p.num_m_tiles * p.num_n_tiles;
  // half-width items exist only for 256-channel tiles
  constexpr bool kHalves = BN == 256;
  const int num_items = kHalves ? pair_num_items(p, num_tiles) : num_tiles;
  const int HW = p.H * p.W;

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], kSP ? 1 : kProd);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 2 * kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    if (p.kchunks_a < p.kchunks) tma_prefetch_desc(&tmA2);
    tma_prefetch_desc(&tmB);
    if (!kDgrad && kHalves && p.half_from < num_tiles) tma_prefetch_desc(&tmB2);
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel's writes are visible from here on
  // rank 0's full and tempty barriers in the cluster window
  const uint32_t full0 = cluster_addr(full, 0);
  const uint32_t tempty0 = cluster_addr(tempty, 0);

  if (warp < kProd) {
    // ------------------------------------------------------------ TMA producers
    // Whole stages in turn (producer `warp` fills the k-blocks issued % kProd
    // == warp), or with KC = 2 every stage's boxes spread over the producers
    // (box b by producer b % kProd): per chunk this CTA's A box, then its
    // weight half.  Rank 0's full barrier counts both CTAs' bytes.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      constexpr int kBPer = (kDgrad || BN == 384) ? Cfg::kDgradBoxes : 1;  // weight boxes per chunk
      constexpr int kPer = 1 + kBPer;
      constexpr int kBoxes = KC * kPer;
      constexpr uint32_t kBBox = (kDgrad || BN == 384) ? 8192u : Cfg::kBHalf;
      // box-parallel: this producer's share of a stage, of a whole tile's and of
      // a half-width item's (half the forward's weight rows; the dgrad's first
      // 64-channel box only)
      uint32_t my_bytes = 0, my_bytes_h = 0;
      for (int b = warp; b < kBoxes; b += kProd) {
        my_bytes += b % kPer == 0 ? kABytes : kBBox;
        my_bytes_h += b % kPer == 0 ? kABytes : kDgrad ? (b % kPer == 1 ? kBBox : 0u) : kBBox / 2;
      }
      constexpr uint32_t kPairStageH = KC * (kABytes + Cfg::kBHalf / 2);
      const int kgroups = p.kchunks / KC;
      for (int it = pair; it < num_items && ok; it += num_pairs) {
        const PairItem w = kHalves ? pair_item(p, it) : PairItem{it, 0, false};
        const int mt = w.tile / p.num_n_tiles, nt = w.tile - mt * p.num_n_tiles;
        const int p0 = mt * 2 * BM + (int)rank * BM;  // this CTA's 128 pixels
        const int n0 = p0 / HW, rem = p0 - n0 * HW;
        const int h0 = rem / p.W;
        const int cn = n0, ch = p.ustride * h0 - 1, cw = p.ustride * (rem - h0 * p.W) - 1;
        // this CTA's weight rows (output channels): half of the tile's, or of the item's 128
        const int c0 = nt * kPairBN + w.coff + (int)rank * (w.half ? 64 : Cfg::kHalf);
        const int kblocks = 9 * kgroups;
        // Box-parallel: rank 1's producers arrive on no barrier, so one with no
        // box in this item's stages (the dgrad's second weight box of a
        // half-width item, or a stage with fewer boxes than producers) gates
        // nothing and could fall two phases behind on its empty barrier, then
        // wait for a phase that never completes: it skips those stages.
        const bool has_boxes = kSP || rank == 0 || (w.half ? my_bytes_h : my_bytes) > 0;
        for (int kb = 0; kb < kblocks; ++kb) {
          const int tap = kb / kgroups, cg = (kb - tap * kgroups) * KC;
          if ((!kSP || issued % kProd == warp) && has_boxes) {
            if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns, p.status, abort_flag)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + (size_t)stage * kPairStage;
            uint8_t* sb = sa + KC * kABytes;
            const uint32_t fb = full0 + (uint32_t)stage * 8u;
            if (rank == 0)
              mbar_arrive_expect_tx(&full[stage], kSP ? 2 * (w.half ? kPairStageH : kPairStage)
                                                      : 2 * (w.half ? my_bytes_h : my_bytes));
            const int wtap = kDgrad ? 8 - tap : tap;
#pragma unroll
            for (int b = 0; b < kBoxes; ++b) {
              if (!kSP && b % kProd != warp) continue;
              const int c = b / kPer, r = b - c * kPer, cc = cg + c;
              if (r == 0) {
                const bool second = cc >= p.kchunks_a;
                tma_load_im2col_4d_pair(sa + c * kABytes, second ? &tmA2 : &tmA, fb,
                                        (second ? cc - p.kchunks_a : cc) * BKC, cw, ch, cn,
                                        (uint16_t)(tap % 3), (uint16_t)(tap / 3));
              } else if constexpr (BN == 384) {
                // channels [128 rank, +128) then [256 + 64 rank, +64) of the tile, as
                // three 64-row (forward) or 64-channel (dgrad) boxes
                const int j = r - 1;
                const int cb = nt * kPairBN + (j < 2 ? 128 * (int)rank + 64 * j : 256 + 64 * (int)rank);
                if (!kDgrad)
                  tma_load_3d_pair(sb + j * 8192, &tmB, fb, cc * BKC, wtap, cb);
                else
                  tma_load_3d_pair(sb + j * 8192, &tmB, fb, cb, wtap, cc * BKC);
              } else if (!kDgrad) {
                // a half-width item's 64 rows come through the 64-row box map
                tma_load_3d_pair(sb + c * Cfg::kBHalf, w.half ? &tmB2 : &tmB, fb, cc * BKC, wtap, c0);
              } else {
                const int j = r - 1;
                if (w.half && j > 0) continue;  // a half-width item takes one 64-channel box
                tma_load_3d_pair(sb + c * Cfg::kBHalf + j * 8192, &tmB, fb, c0 + j * 64, wtap, cc * BKC);
              }
            }
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        if (rank == 0) {
          // wait (bounded) for the loads still in flight
          int n = issued < S ? issued : S;
          int st = stage;
          uint32_t ph = phase;
          for (int i = 0; i < n; ++i) {
            if (--st < 0) {
              st = S - 1;
              ph ^= 1;
            }
            mbar_wait(&full[st], ph, drain_wait_ns(p.wait_ns), nullptr, nullptr);
          }
        } else {
          // rank 1's loads complete on rank 0's barriers: give them time to land
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) __nanosleep(1000);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (rank == 0 && lane == 0) {
      constexpr int kMmaN = BN == 384 ? 256 : kPairBN;  // N = 256 + N = 128 per K step at BN = 384
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, kMmaN, 0, kDgrad ? 1 : 0);
      constexpr uint32_t idesc2 = idesc_bf16_f32(2 * BM, 128, 0, kDgrad ? 1 : 0);  // also half-width items
      // the second MMA's weight rows start after two 8 KB boxes (128 rows or channels)
      constexpr uint32_t kB2 = (2u * 8192u) >> 4;
      const uint32_t sbase = smem_u32(smem);
      const uint64_t a_desc0 = smem_desc(sbase, 16, 1024, kSwizzle128B);
      const uint64_t b_desc0 = kDgrad ? smem_desc(sbase + KC * kABytes, 8192, 1024, kSwizzle128B)
                                      : smem_desc(sbase + KC * kABytes, 16, 1024, kSwizzle128B);
      constexpr uint32_t kStageStep = kPairStage >> 4;
      constexpr uint32_t kBKStep = (kDgrad ? 2048u : 32u) >> 4;
      constexpr uint32_t kAKStep = 32u >> 4;
      int stage = 0;
      uint32_t phase = 0, stage_off = 0;
      int buf = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int it = pair; it < num_items && ok; it += num_pairs) {
        const uint32_t id = (kHalves && it >= p.half_from) ? idesc2 : idesc;
        if (!mbar_wait(&tempty[buf], acc_phase ^ 1, p.wait_ns, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kPairBN);
        const int kblocks = 9 * (p.kchunks / KC);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.wait_ns, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a_desc0 + stage_off, bd = b_desc0 + stage_off;
#pragma unroll
          for (int c = 0; c < KC; ++c)
#pragma unroll
            for (int k = 0; k < BKC / 16; ++k) {
              const uint32_t acc = (kb != 0 || c != 0 || k != 0) ? 1u : 0u;
              tc_mma_bf16_pair(d_tmem, ad + (uint64_t)(c * (kABytes >> 4) + k * kAKStep),
                               bd + (uint64_t)(c * (Cfg::kBHalf >> 4) + k * kBKStep), id, acc);
              if constexpr (BN == 384)
                tc_mma_bf16_pair(d_tmem + 256, ad + (uint64_t)(k * kAKStep), bd + (uint64_t)(kB2 + k * kBKStep),
                                 idesc2, acc);
            }
          tc_commit_pair_mc(&empty[stage], (uint16_t)0x3);
          stage_off += kStageStep;
          if (++stage == S) {
            stage = 0;
            stage_off = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(&tfull[buf], (uint16_t)0x3);
        if (++buf == Cfg::kBufs) {
          buf = 0;
          acc_phase ^= 1;
        }
      }
      // every issued MMA (which reads both CTAs' shared memory and writes both
      // TMEMs) retires before either CTA releases anything
      tc_commit_pair(drain);
      mbar_wait(drain, 0, p.wait_ns, nullptr, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // TMEM lane = this CTA's pixel, column = output channel of the tile (or
    // of the half-width item); the two warps of a lane quarter take half the
    // columns each.
    constexpr int kCols = kPairBN / 2;
    const int q = warp & 3;
    const int half = (warp - kEpiBase) >> 2;
    const int row = q * 32 + lane;
    float* bsl = reinterpret_cast<float*>(smem + (size_t)S * kPairStage + 256) + (warp - kEpiBase) * kCols;
    int buf = 0;
    uint32_t acc_phase = 0;
    for (int it = pair; it < num_items; it += num_pairs) {
      const PairItem w = kHalves ? pair_item(p, it) : PairItem{it, 0, false};
      const int mt = w.tile / p.num_n_tiles, nt = w.tile - mt * p.num_n_tiles;
      const int ncols = kHalves && w.half ? kCols / 2 : kCols;  // this warp's columns
      const int cb = nt * kPairBN + w.coff + half * ncols;     // its first output channel
      const long long pix = (long long)mt * 2 * BM + rank * BM + row;
      const bool valid = pix < p.P;
      if (kExt && kDgrad && p.zin && valid && cb < p.nout) prefetch_zin_row(p, pix, cb, ncols);
      if (!kDgrad && p.bias) stage_bias_slice<kCols>(p, cb, bsl, lane);
      if (!mbar_wait(&tfull[buf], acc_phase, p.wait_ns, p.status, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kPairBN + half * ncols);
      // every item of one-item pairs (epi_tma 1) or each pair's last item
      // (epi_tma 2) leaves through TMA stores staged in the idle stage rings
      const bool tma_here = p.epi_tma == 1 || (p.epi_tma == 2 && it + num_pairs >= num_items);
      if constexpr (kCols % 64 == 0) {
        if (tma_here) {
          // both stage rings are idle (every MMA of the tile has completed);
          // this warp's 32 pixels leave as ncols / 64 boxes of {64 channels, 32 pixels}
          uint8_t* stg = smem + (size_t)(warp - kEpiBase) * (kCols / 64) * 4096u;
          const long long wrow0 = (long long)mt * 2 * BM + rank * BM + q * 32;
#pragma unroll 1
          for (int j = 0; j < ncols / 32; ++j) {
            const int col0 = cb + j * 32;
            float bv[32];
            if (!kDgrad && p.bias) bias_from_slice(bsl + j * 32, bv);
            uint4 zr[4] = {};
            if (kExt && kDgrad && p.zin && valid && col0 < p.nout) load_zin(p, pix, col0, zr);
            uint32_t v[32];
            tmem_ld_32x32b_x32(taddr + (uint32_t)(j * 32), v);
            tmem_ld_wait();
            uint8_t* box = stg + (j >> 1) * 4096u;
            stage_chunk_bf16<kExt, kDgrad ? 1 : 0>(p, v, bv, zr, box + lane * 128, (j & 1) * 4, lane);
            if (j & 1) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0 && col0 - 32 < p.nout && wrow0 < p.P) tma_store_2d(&tmY, box, col0 - 32, (int)wrow0);
            }
          }
          if (lane == 0) {
            bulk_commit();
            bulk_wait_read<0>();  // the stores' writes complete with the grid
          }
          __syncwarp();
        }
      }
#pragma unroll 1
      for (int j = 0; j < (tma_here && kCols % 64 == 0 ? 0 : ncols / 32); ++j) {
        const int col0 = cb + j * 32;
        const bool live = valid && col0 < p.nout;
        float bv[32];
        if (!kDgrad && p.bias && live) bias_from_slice(bsl + j * 32, bv);
        uint4 zr[4] = {};
        if (kExt && kDgrad && p.zin && live) load_zin(p, pix, col0, zr);
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + (uint32_t)(j * 32), v);
        tmem_ld_wait();
        if (live) store_chunk<kExt, kDgrad ? 1 : 0>(p, pix, col0, v, bv, zr);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + (uint32_t)buf * 8u);
      if (++buf == Cfg::kBufs) {
        buf = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc_pair(tmem_base, 512);
}

// ----------------------------------------------------------------------------
// forward / dgrad with each tile's K split over a two-CTA cluster
// ----------------------------------------------------------------------------
// For grids that leave most of the GPU idle with 256-channel tiles (the 8x8
// layers: 4096 pixels x 512 channels are 64 tiles of 128 x 256).  A cluster of
// two CTAs owns one 128-pixel x 256-channel tile; rank r runs k-blocks
// [r h, r h + h) of its K (h = half the 9 x chunks k-blocks) with one-CTA
// N = 256 MMAs -- four per barrier round trip of the issuing thread where the
// 128 x 128 tiles these grids otherwise take issue eight N = 128 MMAs -- into a
// 256-column accumulator.  The two accumulators are then added through
// distributed shared memory: each CTA writes the 128 columns the peer stores
// into the peer's (then idle) stage memory, as [column / 4][pixel] float4s so
// that a warp's 16-byte stores and loads are contiguous, and each CTA adds the
// received half to its own and stores it.  Both CTAs add the same two fp32
// values, so the result does not depend on which one stores a column.  Two
// cluster barriers, passed by every thread on every path (an aborted role
// still reaches them), order the exchange.
constexpr int kKsBN = 256;
constexpr uint32_t kKsStage = kABytes + kKsBN * 128;  // 128-pixel A box + 256 weight rows x 64 channels
constexpr int kKsStages = 4;
constexpr uint32_t kKsXchg = 128u * 128u * 4u;        // 128 pixels x 128 fp32 columns
// + barriers, + the epilogue warps' bias slices (64 columns each), + slack
constexpr size_t kKsSmem = (size_t)kKsStages * kKsStage + 256 + kEpiWarps * 64 * 4 + 1024 + kGuardBytes;
static_assert(kKsSmem <= 227 * 1024, "shared memory per CTA");
static_assert(kKsXchg <= (uint32_t)kKsStages * kKsStage, "the exchange reuses the stage memory");
static_assert(kKsStages >= kProd, "stage-parallel producers need S >= kProd");

template <bool kDgrad, bool kExt>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kIgemmThreads, 1)
    k_igemm_ks(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
               const __grid_constant__ CUtensorMap tmB, const IgemmParams p) {
  constexpr int S = kKsStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * kKsStage);
  uint64_t* empty = full + S;
  uint64_t* drain = empty + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  const uint32_t rank = cluster_ctarank();
  const int tile = blockIdx.x >> 1;
  const int mt = tile / p.num_n_tiles, nt = tile - mt * p.num_n_tiles;
  const int HW = p.H * p.W;
  const int kb_total = 9 * p.kchunks;
  const int kb_half = (kb_total + 1) / 2;
  const int kb0 = (int)rank * kb_half;
  const int kb1 = min(kb_total, kb0 + kb_half);

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    if (p.kchunks_a < p.kchunks) tma_prefetch_desc(&tmA2);
    tma_prefetch_desc(&tmB);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kKsBN);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel's writes are visible from here on
  // epilogue warp ew stores columns 128 rank + 64 ((ew >> 2) & 1) .. + 63:
  // their bias is staged while the main loop runs
  float* bsl = reinterpret_cast<float*>(smem + (size_t)S * kKsStage + 256) + (warp - kEpiBase) * 64;
  if (warp >= kEpiBase && !kDgrad && p.bias)
    stage_bias_slice<64>(p, nt * kKsBN + 128 * (int)rank + 64 * (((warp - kEpiBase) >> 2) & 1), bsl, lane);

  if (warp < kProd) {
    // whole stages in turn: the A box and the weight tile (one 256-row box,
    // or four 64-channel MN-major boxes for dgrad)
    if (lane == 0) {
      const int p0 = mt * BM;
      const int n0 = p0 / HW, rem = p0 - n0 * HW;
      const int h0 = rem / p.W;
      const int cn = n0, ch = p.ustride * h0 - 1, cw = p.ustride * (rem - h0 * p.W) - 1;
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (issued % kProd == warp) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns, p.status, abort_flag)) {
            ok = false;
            break;
          }
          const int tap = kb / p.kchunks, cc = kb - tap * p.kchunks;
          uint8_t* sa = smem + (size_t)stage * kKsStage;
          uint8_t* sb = sa + kABytes;
          mbar_arrive_expect_tx(&full[stage], kKsStage);
          const bool second = cc >= p.kchunks_a;
          tma_load_im2col_4d(sa, second ? &tmA2 : &tmA, &full[stage], (second ? cc - p.kchunks_a : cc) * BKC, cw,
                             ch, cn, (uint16_t)(tap % 3), (uint16_t)(tap / 3));
          const int wtap = kDgrad ? 8 - tap : tap;
          if (!kDgrad) {
            tma_load_3d(sb, &tmB, &full[stage], cc * BKC, wtap, nt * kKsBN);
          } else {
#pragma unroll
            for (int j = 0; j < kKsBN / 64; ++j)
              tma_load_3d(sb + j * 8192, &tmB, &full[stage], nt * kKsBN + j * 64, wtap, cc * BKC);
          }
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        int n = issued < S ? issued : S;
        for (int i = 0; i < n; ++i) {
          if (--stage < 0) {
            stage = S - 1;
            phase ^= 1;
          }
          mbar_wait(&full[stage], phase, drain_wait_ns(p.wait_ns), nullptr, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, kKsBN, 0, kDgrad ? 1 : 0);
      const uint32_t sbase = smem_u32(smem);
      const uint64_t a_desc0 = smem_desc(sbase, 16, 1024, kSwizzle128B);
      const uint64_t b_desc0 = kDgrad ? smem_desc(sbase + kABytes, 8192, 1024, kSwizzle128B)
                                      : smem_desc(sbase + kABytes, 16, 1024, kSwizzle128B);
      constexpr uint32_t kStageStep = kKsStage >> 4;
      constexpr uint32_t kBKStep = (kDgrad ? 2048u : 32u) >> 4;
      constexpr uint32_t kAKStep = 32u >> 4;
      int stage = 0;
      uint32_t phase = 0, stage_off = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full[stage], phase, p.wait_ns, p.status, abort_flag)) break;
        tc_fence_after();
        const uint64_t ad = a_desc0 + stage_off, bd = b_desc0 + stage_off;
#pragma unroll
        for (int k = 0; k < BKC / 16; ++k)
          tc_mma_bf16(tmem_base, ad + (uint64_t)(k * kAKStep), bd + (uint64_t)(k * kBKStep), idesc,
                      (kb != kb0 || k != 0) ? 1u : 0u);
        tc_commit(&empty[stage]);
        stage_off += kStageStep;
        if (++stage == S) {
          stage = 0;
          stage_off = 0;
          phase ^= 1;
        }
      }
      // every MMA has completed before the cluster barrier below
      tc_commit(drain);
      mbar_wait(drain, 0, p.wait_ns, nullptr, nullptr);
    }
    __syncwarp();
  }

  // both CTAs' accumulators are complete and their stage memory idle
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const int ew = warp - kEpiBase;
  const int q = warp & 3;
  const int hw = (ew >> 2) & 1;  // which 64 of the CTA's 128 exchanged / stored columns
  const int row = q * 32 + lane;
  const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
  const bool run = warp >= kEpiBase && !*abort_flag;
  if (run) {
    // send the peer's columns [128 (rank ^ 1) + 64 hw, +64) into its stage memory
    const uint32_t peer_buf = cluster_addr(smem, rank ^ 1u);
#pragma unroll 1
    for (int j = 0; j < 2; ++j) {
      const int cl = hw * 64 + j * 32;  // column within the peer's half
      uint32_t v[32];
      tmem_ld_32x32b_x32(lane_addr + (uint32_t)(128 * (rank ^ 1u) + cl), v);
      tmem_ld_wait();
#pragma unroll
      for (int g = 0; g < 8; ++g)
        st_cluster_v4(peer_buf + (uint32_t)(((cl / 4 + g) * 128 + row) * 16), v[4 * g], v[4 * g + 1], v[4 * g + 2],
                      v[4 * g + 3]);
    }
  }
  // the received columns are visible once every thread passes here
  __syncwarp();
  cluster_sync();
  if (run) {
    const long long pix = (long long)mt * BM + row;
    const bool valid = pix < p.P;
    const uint4* recv = reinterpret_cast<const uint4*>(smem);
#pragma unroll 1
    for (int j = 0; j < 2; ++j) {
      const int cl = hw * 64 + j * 32;  // column within this CTA's half
      const int col0 = nt * kKsBN + 128 * (int)rank + cl;
      const bool live = valid && col0 < p.nout;
      float bv[32];
      if (!kDgrad && p.bias && live) bias_from_slice(bsl + j * 32, bv);
      uint4 zr[4] = {};
      if (kExt && kDgrad && p.zin && live) load_zin(p, pix, col0, zr);
      uint32_t v[32];
      tmem_ld_32x32b_x32(lane_addr + (uint32_t)(128 * rank + cl), v);
      tmem_ld_wait();
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const uint4 r = recv[(cl / 4 + g) * 128 + row];
        v[4 * g] = __float_as_uint(__uint_as_float(v[4 * g]) + __uint_as_float(r.x));
        v[4 * g + 1] = __float_as_uint(__uint_as_float(v[4 * g + 1]) + __uint_as_float(r.y));
        v[4 * g + 2] = __float_as_uint(__uint_as_float(v[4 * g + 2]) + __uint_as_float(r.z));
        v[4 * g + 3] = __float_as_uint(__uint_as_float(v[4 * g + 3]) + __uint_as_float(r.w));
      }
      if (live) store_chunk<kExt, kDgrad ? 1 : 0>(p, pix, col0, v, bv, zr);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, kKsBN);
}

// ----------------------------------------------------------------------------
// forward / dgrad: 256-pixel x 256-channel pair tiles with K split over two
// pairs (clusters of four CTAs)
// ----------------------------------------------------------------------------
// For grids too small for whole pair tiles (the 8x8 layers: 4096 pixels x 512
// channels are 32 tiles of 256 x 256, 64 CTAs).  Ranks 0-1 and 2-3 of a
// cluster are two CTA pairs (tcgen05 cta_group::2, peers differ in rank bit
// 0); pair h = rank >> 1 runs the tile's k-blocks [h kh, h kh + kh) with the
// M = 256, N = 256 MMAs of k_igemm_pair (two 64-channel chunks per stage: each
// CTA streams 32 KB per 1024 cycles of tensor work), so the tile's 128 CTAs
// fill most of the GPU.  Each CTA then holds its 128 pixels x 256 channels of
// one K half.  The two CTAs with the same pixels (ranks r and r ^ 2) add them
// through distributed shared memory as k_igemm_ks does: each writes the 128
// columns the other stores into the other's (then idle) stage memory, then
// adds the received half to its own and stores it; both add the same two fp32
// values in the same order, so a column's sum does not depend on which CTA
// stores it.  Every wait is bounded; the cluster barriers are reached by
// every thread on every path.
constexpr int kPksBN = 256;
constexpr int kPksKC = 2;

template <bool kDgrad, bool kExt>
__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kIgemmThreads, 1)
    k_igemm_pks(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                const __grid_constant__ CUtensorMap tmB, const IgemmParams p) {
  using Cfg = PairCfg<kPksBN, kDgrad, kPksKC>;
  constexpr int S = Cfg::kStages;
  constexpr int KC = kPksKC;
  constexpr uint32_t kStageBytes = Cfg::kStage;
  static_assert((uint32_t)S * Cfg::kStage >= 128u * 128u * 4u, "the exchange reuses the stage memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* drain = empty + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  const uint32_t rank = cluster_ctarank();
  const uint32_t pr = rank & 1u;        // pixel half within the pair
  const uint32_t h = rank >> 1;         // K half
  const uint32_t leader = rank & ~1u;   // the pair's MMA-issuing CTA
  const int tile = blockIdx.x >> 2;
  const int mt = tile / p.num_n_tiles, nt = tile - mt * p.num_n_tiles;
  const int HW = p.H * p.W;
  const int kb_total = 9 * (p.kchunks / KC);
  const int kb_half = (kb_total + 1) / 2;
  const int kb0 = (int)h * kb_half;
  const int kb1 = min(kb_total, kb0 + kb_half);

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], Cfg::kSP ? 1 : kProd);
      mbar_init(&empty[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    if (p.kchunks_a < p.kchunks) tma_prefetch_desc(&tmA2);
    tma_prefetch_desc(&tmB);
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(tmem_slot, kPksBN);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel's writes are visible from here on
  const uint32_t full_l = cluster_addr(full, leader);
  // epilogue warp ew stores columns 128 h + 64 ((ew >> 2) & 1) .. + 63: their
  // bias is staged while the main loop runs
  float* bsl = reinterpret_cast<float*>(smem + (size_t)S * kStageBytes + 256) + (warp - kEpiBase) * 64;
  if (warp >= kEpiBase && !kDgrad && p.bias)
    stage_bias_slice<64>(p, nt * kPksBN + 128 * (int)h + 64 * (((warp - kEpiBase) >> 2) & 1), bsl, lane);

  if (warp < kProd) {
    // as k_igemm_pair: per chunk this CTA's A box, then its 128 weight rows
    // (one box forward, two 64-channel boxes dgrad); the leader's full barrier
    // counts both CTAs' bytes
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      constexpr int kBPer = kDgrad ? Cfg::kDgradBoxes : 1;
      constexpr int kPer = 1 + kBPer;
      constexpr int kBoxes = KC * kPer;
      constexpr uint32_t kBBox = kDgrad ? 8192u : Cfg::kBHalf;
      uint32_t my_bytes = 0;
      for (int b = warp; b < kBoxes; b += kProd) my_bytes += b % kPer == 0 ? kABytes : kBBox;
      const int kgroups = p.kchunks / KC;
      const int p0 = mt * 2 * BM + (int)pr * BM;  // this CTA's 128 pixels
      const int n0 = p0 / HW, rem = p0 - n0 * HW;
      const int h0 = rem / p.W;
      const int cn = n0, ch = p.ustride * h0 - 1, cw = p.ustride * (rem - h0 * p.W) - 1;
      const int c0 = nt * kPksBN + (int)pr * Cfg::kHalf;  // this CTA's weight rows
      // (as in k_igemm_pair: a second-rank producer without boxes skips the stages)
      const bool has_boxes = Cfg::kSP || pr == 0 || my_bytes > 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        const int tap = kb / kgroups, cg = (kb - tap * kgroups) * KC;
        if ((!Cfg::kSP || issued % kProd == warp) && has_boxes) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns, p.status, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * kStageBytes;
          uint8_t* sb = sa + KC * kABytes;
          const uint32_t fb = full_l + (uint32_t)stage * 8u;
          if (pr == 0) mbar_arrive_expect_tx(&full[stage], Cfg::kSP ? 2 * kStageBytes : 2 * my_bytes);
          const int wtap = kDgrad ? 8 - tap : tap;
#pragma unroll
          for (int b = 0; b < kBoxes; ++b) {
            if (!Cfg::kSP && b % kProd != warp) continue;
            const int c = b / kPer, r = b - c * kPer, cc = cg + c;
            if (r == 0) {
              const bool second = cc >= p.kchunks_a;
              tma_load_im2col_4d_pair(sa + c * kABytes, second ? &tmA2 : &tmA, fb,
                                      (second ? cc - p.kchunks_a : cc) * BKC, cw, ch, cn, (uint16_t)(tap % 3),
                                      (uint16_t)(tap / 3));
            } else if (!kDgrad) {
              tma_load_3d_pair(sb + c * Cfg::kBHalf, &tmB, fb, cc * BKC, wtap, c0);
            } else {
              const int j = r - 1;
              tma_load_3d_pair(sb + c * Cfg::kBHalf + j * 8192, &tmB, fb, c0 + j * 64, wtap, cc * BKC);
            }
          }
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        if (pr == 0) {
          // wait (bounded) for the loads still in flight
          int n = issued < S ? issued : S;
          int st = stage;
          uint32_t ph = phase;
          for (int i = 0; i < n; ++i) {
            if (--st < 0) {
              st = S - 1;
              ph ^= 1;
            }
            mbar_wait(&full[st], ph, drain_wait_ns(p.wait_ns), nullptr, nullptr);
          }
        } else {
          // the peer's loads complete on the leader's barriers: give them time to land
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) __nanosleep(1000);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (the pair's leader)
    if (pr == 0 && lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, kPksBN, 0, kDgrad ? 1 : 0);
      const uint32_t sbase = smem_u32(smem);
      const uint64_t a_desc0 = smem_desc(sbase, 16, 1024, kSwizzle128B);
      const uint64_t b_desc0 = kDgrad ? smem_desc(sbase + KC * kABytes, 8192, 1024, kSwizzle128B)
                                      : smem_desc(sbase + KC * kABytes, 16, 1024, kSwizzle128B);
      constexpr uint32_t kStageStep = kStageBytes >> 4;
      constexpr uint32_t kBKStep = (kDgrad ? 2048u : 32u) >> 4;
      constexpr uint32_t kAKStep = 32u >> 4;
      const uint16_t mask = (uint16_t)(0x3u << leader);  // both CTAs of this pair
      int stage = 0;
      uint32_t phase = 0, stage_off = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full[stage], phase, p.wait_ns, p.status, abort_flag)) break;
        tc_fence_after();
        const uint64_t ad = a_desc0 + stage_off, bd = b_desc0 + stage_off;
#pragma unroll
        for (int c = 0; c < KC; ++c)
#pragma unroll
          for (int k = 0; k < BKC / 16; ++k)
            tc_mma_bf16_pair(tmem_base, ad + (uint64_t)(c * (kABytes >> 4) + k * kAKStep),
                             bd + (uint64_t)(c * (Cfg::kBHalf >> 4) + k * kBKStep), idesc,
                             (kb != kb0 || c != 0 || k != 0) ? 1u : 0u);
        tc_commit_pair_mc(&empty[stage], mask);
        stage_off += kStageStep;
        if (++stage == S) {
          stage = 0;
          stage_off = 0;
          phase ^= 1;
        }
      }
      // every issued MMA (which reads both CTAs' shared memory and writes both
      // TMEMs) retires before the cluster barrier below
      tc_commit_pair(drain);
      mbar_wait(drain, 0, p.wait_ns, nullptr, nullptr);
    }
    __syncwarp();
  }

  // all four CTAs' accumulators are complete and their stage memory idle
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const int ew = warp - kEpiBase;
  const int q = warp & 3;
  const int hw = (ew >> 2) & 1;  // which 64 of the CTA's 128 exchanged / stored columns
  const int row = q * 32 + lane;
  const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
  const bool run = warp >= kEpiBase && !*abort_flag;
  if (run) {
    // send the partner's columns [128 (h ^ 1) + 64 hw, +64) into its stage memory
    const uint32_t peer_buf = cluster_addr(smem, rank ^ 2u);
#pragma unroll 1
    for (int j = 0; j < 2; ++j) {
      const int cl = hw * 64 + j * 32;  // column within the partner's half
      uint32_t v[32];
      tmem_ld_32x32b_x32(lane_addr + (uint32_t)(128 * (h ^ 1u) + cl), v);
      tmem_ld_wait();
#pragma unroll
      for (int g = 0; g < 8; ++g)
        st_cluster_v4(peer_buf + (uint32_t)(((cl / 4 + g) * 128 + row) * 16), v[4 * g], v[4 * g + 1], v[4 * g + 2],
                      v[4 * g + 3]);
    }
  }
  // the received columns are visible once every thread passes here
  __syncwarp();
  cluster_sync();
  if (run) {
    const long long pix = (long long)mt * 2 * BM + (long long)pr * BM + row;
    const bool valid = pix < p.P;
    const uint4* recv = reinterpret_cast<const uint4*>(smem);
#pragma unroll 1
    for (int j = 0; j < 2; ++j) {
      const int cl = hw * 64 + j * 32;  // column within this CTA's half
      const int col0 = nt * kPksBN + 128 * (int)h + cl;
      const bool live = valid && col0 < p.nout;
      float bv[32];
      if (!kDgrad && p.bias && live) bias_from_slice(bsl + j * 32, bv);
      uint4 zr[4] = {};
      if (kExt && kDgrad && p.zin && live) load_zin(p, pix, col0, zr);
      uint32_t v[32];
      tmem_ld_32x32b_x32(lane_addr + (uint32_t)(128 * h + cl), v);
      tmem_ld_wait();
      // own K half + the partner's (one fp32 addition per element: the same
      // sum whichever CTA forms it)
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const uint4 r = recv[(cl / 4 + g) * 128 + row];
        v[4 * g] = __float_as_uint(__uint_as_float(v[4 * g]) + __uint_as_float(r.x));
        v[4 * g + 1] = __float_as_uint(__uint_as_float(v[4 * g + 1]) + __uint_as_float(r.y));
        v[4 * g + 2] = __float_as_uint(__uint_as_float(v[4 * g + 2]) + __uint_as_float(r.z));
        v[4 * g + 3] = __float_as_uint(__uint_as_float(v[4 * g + 3]) + __uint_as_float(r.w));
      }
      if (live) store_chunk<kExt, kDgrad ? 1 : 0>(p, pix, col0, v, bv, zr);
    }
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc_pair(tmem_base, kPksBN);
}

// ----------------------------------------------------------------------------
// forward / dgrad implicit GEMM, halo variant (image widths 16, 32, 64)
// ----------------------------------------------------------------------------
// A CTA tile is R = 256 / W whole image rows (256 output pixels, two 128-row
// MMAs per k-step).  For each 64-channel chunk and column shift s in {0,1,2}
// one tiled TMA box holds the R + 2 zero-padded input rows h0-1 .. h0+R at
// columns s-1 .. s-2+W; it serves all three row taps r, whose A operand is the
// same box from row r*W on (a 1024-byte-aligned offset).  Every input pixel is
// staged three times per chunk instead of nine.  A boxes and weight tiles
// stream through separate rings; producer warps 0-1 load the two halves of
// each A box, warps 2-3 the 64-row halves of each weight tile.
template <int W_, int BN>
struct HaloCfg {
  static constexpr int R = 256 / W_;
  static constexpr int kHalfRows = (R + 2) / 2;
  static constexpr uint32_t kABytes = (uint32_t)(R + 2) * W_ * 128;
  static constexpr uint32_t kAHalfBytes = kABytes / 2;
  static constexpr uint32_t kBBytes = BN * 128;
  static constexpr int kSA = 3;
  static constexpr int kSBFit = (int)((208u * 1024u - kSA * kABytes) / kBBytes);
  static constexpr int kSB = kSBFit > 8 ? 8 : kSBFit;
  static constexpr int kTmemCols = pow2_cols(4 * BN);
  static constexpr size_t kSmem = (size_t)kSA * kABytes + (size_t)kSB * kBBytes + 512 + 1024 + 8 * 1024;
  static_assert((R + 2) % 2 == 0 && kAHalfBytes % 1024 == 0, "A halves must stay swizzle-atom aligned");
  static_assert(kSB >= 3, "weight ring too shallow");
};

template <int W_, int BN, bool kDgrad>
__global__ void __launch_bounds__(kIgemmThreads, 1)
    k_halo(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const IgemmParams p) {
  using Cfg = HaloCfg<W_, BN>;
  constexpr int SA = Cfg::kSA, SB = Cfg::kSB, TM = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* ringA = smem;
  uint8_t* ringB = smem + (size_t)SA * Cfg::kABytes;
  uint64_t* fullA = reinterpret_cast<uint64_t*>(ringB + (size_t)SB * Cfg::kBBytes);
  uint64_t* emptyA = fullA + SA;
  uint64_t* fullB = emptyA + SA;
  uint64_t* emptyB = fullB + SB;
  uint64_t* tfull = emptyB + SB;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  const int num_tiles = p.num_m_tiles * p.num_n_tiles;
  const int HW = p.H * W_;

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < SA; ++i) {
      mbar_init(&fullA[i], 2);
      mbar_init(&emptyA[i], 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&fullB[i], 2);
      mbar_init(&emptyB[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel's writes are visible from here on

  if (warp < 2) {
    // ------------------------------------------------------------ A-box producers
    if (lane == 0) {
      int st = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int mt = tile / p.num_n_tiles;
        const int p0 = mt * TM;
        const int n0 = p0 / HW, h0 = (p0 - n0 * HW) / W_;
        for (int cc = 0; cc < p.kchunks && ok; ++cc)
          for (int s = 0; s < 3; ++s) {
            if (!mbar_wait(&emptyA[st], ph ^ 1, p.wait_ns, p.status, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&fullA[st], Cfg::kAHalfBytes);
            tma_load_4d(ringA + (size_t)st * Cfg::kABytes + warp * Cfg::kAHalfBytes, &tmA, &fullA[st],
                        cc * BKC, s - 1, h0 - 1 + warp * Cfg::kHalfRows, n0);
            ++issued;
            if (++st == SA) {
              st = 0;
              ph ^= 1;
            }
          }
      }
      if (!ok) {
        int n = issued < SA ? issued : SA;
        for (int i = 0; i < n; ++i) {
          if (--st < 0) {
            st = SA - 1;
            ph ^= 1;
          }
          mbar_wait(&fullA[st], ph, drain_wait_ns(p.wait_ns), nullptr, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp < kProd) {
    // ------------------------------------------------------------ weight producers
    if (lane == 0) {
      const int j = warp - 2;  // 64-row half of the weight tile
      const bool loads = j < BN / 64;
      int st = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int nt = tile % p.num_n_tiles;
        for (int cc = 0; cc < p.kchunks && ok; ++cc)
          for (int s = 0; s < 3 && ok; ++s)
            for (int r = 0; r < 3; ++r) {
              if (!mbar_wait(&emptyB[st], ph ^ 1, p.wait_ns, p.status, abort_flag)) {
                ok = false;
                break;
              }
              const int tap = 3 * r + s;
              mbar_arrive_expect_tx(&fullB[st], loads ? 8192u : 0u);
              if (loads) {
                uint8_t* dst = ringB + (size_t)st * Cfg::kBBytes + j * 8192;
                if (!kDgrad)
                  tma_load_3d(dst, &tmB, &fullB[st], cc * BKC, tap, nt * BN + j * 64);
                else
                  tma_load_3d(dst, &tmB, &fullB[st], nt * BN + j * 64, 8 - tap, cc * BKC);
              }
              ++issued;
              if (++st == SB) {
                st = 0;
                ph ^= 1;
              }
            }
      }
      if (!ok) {
        int n = issued < SB ? issued : SB;
        for (int i = 0; i < n; ++i) {
          if (--st < 0) {
            st = SB - 1;
            ph ^= 1;
          }
          mbar_wait(&fullB[st], ph, drain_wait_ns(p.wait_ns), nullptr, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0, kDgrad ? 1 : 0);
      int sa = 0, sb = 0, buf = 0;
      uint32_t pa = 0, pb = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        if (!mbar_wait(&tempty[buf], acc_phase ^ 1, p.wait_ns, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * 2 * BN);
        bool first = true;
        for (int cc = 0; cc < p.kchunks && ok; ++cc)
          for (int s = 0; s < 3 && ok; ++s) {
            if (!mbar_wait(&fullA[sa], pa, p.wait_ns, p.status, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(ringA + (size_t)sa * Cfg::kABytes);
            for (int r = 0; r < 3; ++r) {
              if (!mbar_wait(&fullB[sb], pb, p.wait_ns, p.status, abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t b_base = smem_u32(ringB + (size_t)sb * Cfg::kBBytes);
#pragma unroll
              for (int k = 0; k < BKC / 16; ++k) {
                const uint64_t bdesc = kDgrad ? smem_desc(b_base + k * 2048, 8192, 1024, kSwizzle128B)
                                              : smem_desc(b_base + k * 32, 16, 1024, kSwizzle128B);
#pragma unroll
                for (int u = 0; u < 2; ++u)
                  tc_mma_bf16(d_tmem + (uint32_t)(u * BN),
                              smem_desc(a_base + (uint32_t)(u * BM + r * W_) * 128 + k * 32, 16, 1024,
                                        kSwizzle128B),
                              bdesc, idesc, (first && k == 0) ? 0u : 1u);
              }
              first = false;
              tc_commit(&emptyB[sb]);
              if (++sb == SB) {
                sb = 0;
                pb ^= 1;
              }
            }
            if (!ok) break;
            tc_commit(&emptyA[sa]);
            if (++sa == SA) {
              sa = 0;
              pa ^= 1;
            }
          }
        if (!ok) break;
        tc_commit(&tfull[buf]);
        if (++buf == 2) {
          buf = 0;
          acc_phase ^= 1;
        }
      }
      tc_commit(drain);
      mbar_wait(drain, 0, p.wait_ns, nullptr, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int sub = (warp - kEpiBase) >> 2;  // 128-pixel half of the tile
    const int row = q * 32 + lane;
    int buf = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      if (!mbar_wait(&tfull[buf], acc_phase, p.wait_ns, p.status, abort_flag)) break;
      tc_fence_after();
      const int mt = tile / p.num_n_tiles, nt = tile % p.num_n_tiles;
      const long long pix = (long long)mt * TM + sub * BM + row;
      const bool valid = pix < p.P;
      const uint32_t taddr =
          tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)((buf * 2 + sub) * BN);
#pragma unroll 1
      for (int j = 0; j < BN / 32; ++j) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + (uint32_t)(j * 32), v);
        tmem_ld_wait();
        const int col0 = nt * BN + j * 32;
        if (valid && col0 < p.nout) store_chunk(p, pix, col0, v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      if (++buf == 2) {
        buf = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, Cfg::kTmemCols);
}

// ----------------------------------------------------------------------------
// forward, 8 input channels (the UNet stem: RGB zero-padded to 8)
// ----------------------------------------------------------------------------
// With 8 channels a tap is 16 bytes per pixel, so a 64-channel SW128 k-block
// would be seven-eighths zero fill.  Here each tap is one im2col box of 128
// pixels x 8 channels (2 KB, no swizzle): in the K-major no-swizzle operand
// layout that box is exactly a column of 8x16-byte core matrices, and taps
// 2j, 2j+1 form the K = 16 of MMA j (K = 9 taps x 8 + one zero tap = 80, five
// MMAs per tile).  The weights ([Cout][9][8], 2 KB per tap for 128 outputs) stay
// resident in shared memory for the whole kernel.
//
// The bias rides in the padding tap: its A block holds 1.0 in channels 0 and 1
// for every pixel, its weight row k holds bias[k] split into two bf16 parts
// (hi = RNE(bias), lo = RNE(bias - hi), together exact to 2^-18 relative), so
// the accumulator comes out of the tensor core as conv + bias and the epilogue
// -- this kernel's bottleneck -- only applies the activation (SiLU through
// tanh, one special-function op) and rounds.
//
// kTS (BN = 128, bf16 y, no z store): the output leaves through TMA stores.
// Each epilogue warp owns 32 pixels x 64 channels of a tile -- 32 rows of
// 128 bytes, contiguous rows of y -- which it stages in shared memory in the
// 128-byte-swizzled layout of a {64 channels, 32 pixels} box (16-byte chunk c
// of row r at chunk c ^ (r % 8): the eight rows a store phase covers hit all
// 32 banks) and hands to one TMA tensor store; two staging buffers per warp let
// a tile's stores overlap the next tile's epilogue.  The direct path writes the
// same bytes as per-thread 16-byte stores spread over 32 pixel rows.
//
// kRW (image width 32 or 64, whole-row tiles): x staged in long rows instead
// of im2col boxes.  An im2col box of 8 channels moves 128 rows of 16 bytes, and
// the copy engine's row rate -- not bytes -- set this kernel's pace.  Viewing x
// as [N][H][W * 8], an image row is one run of W * 16 bytes; for each column
// shift s the stage holds a slot of the tile's R = 128 / W image rows plus the
// row above and below, shifted by s - 1 pixels (the columns and rows outside
// the image read zero), in 512-byte boxes.  Tap (r, s) -- K slot q = 3 s + r --
// is then the 128 pixels that start r rows into slot s: 24 (W = 64) or 18
// (W = 32) copy rows per tile instead of 1152.  The weights sit in the same
// slot order.
template <int BN, bool kTS = false, int kRW = 0, bool kZ = false>
struct StemCfg {
  static constexpr uint32_t kTapBytes = BM * 16;           // 128 pixels x 8 channels
  static constexpr int kRowsPerTile = kRW ? BM / kRW : 0;  // image rows of a tile (kRW)
  static constexpr uint32_t kRowBytes = (uint32_t)kRW * 16;  // one image row of x (kRW)
  static constexpr uint32_t kSlotBytes = (uint32_t)(kRowsPerTile + 2) * kRowBytes;
  static constexpr int kBoxElems = kRW * 8 < 256 ? kRW * 8 : 256;  // elements per row box
  static constexpr int kRowParts = kRW ? kRW * 8 / kBoxElems : 0;  // boxes per image row
  // A offset of the tenth (padding) K slot: after the 9 taps, or the 3 slots
  static constexpr uint32_t kPadOff = kRW ? 3 * kSlotBytes : 9 * kTapBytes;
  static constexpr uint32_t kStageBytes = kPadOff + kTapBytes;  // + padding tap
  static constexpr uint32_t kBTap = BN * 16;
  static constexpr uint32_t kBBytes = 10 * kBTap;
  // kZ (TMA-store epilogue only): z = conv + bias leaves through TMA stores
  // too, from a second set of staging boxes, with four stages
  static constexpr int kStages = kTS ? (kZ ? 4 : kRW ? 8 : 6) : 8;
  static constexpr uint32_t kStageOutBytes = 32 * 128;     // one warp's 32 x 64 bf16 box
  static constexpr uint32_t kOutBytes = kTS ? (kZ ? 2 : 1) * 2 * kEpiWarps * kStageOutBytes : 0;
  static constexpr int kTmemCols = pow2_cols(2 * BN);
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + kBBytes + kOutBytes + 512 + 1024;
  static_assert(kStages >= kProd, "stage-parallel producers need S >= kProd");
  static_assert(!kTS || BN == 128, "the TMA-store epilogue covers 128-channel tiles");
  static_assert(!kZ || (kTS && kRW != 0), "z through TMA stores with row staging only");
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
  static_assert(((size_t)kStages * kStageBytes + kBBytes) % 1024 == 0, "staging must be 1 KB aligned");
  static_assert(kRW == 0 || kRW == 32 || kRW == 64, "row staging for widths 32 and 64");
};

// Byte offset in the A stage of K slot q (0..8: taps in the stage's order,
// 9: the padding tap).  im2col: slot q holds tap q; row staging: slot q holds
// tap (q % 3) * 3 + q / 3 (r = q % 3 rows into the slot of shift s = q / 3).
// The stem's resident B operand: K slot q (0..8) holds one tap of every output
// channel as a 16-byte row (rows at or past nout zero), slot 9 the bias split
// into two bf16 halves (hi, lo) in channels 0-1.  Slot q holds tap q, or with
// row staging (kRW) tap 3 (q % 3) + q / 3.  Run by the kEpiWarps epilogue
// warps (t = 0 .. 32 kEpiWarps - 1): coalesced 16-byte loads in w's own order
// [Cout][9][8], then one arrival per warp on `ready`.  Nine TMA boxes of
// 16-byte rows took ~4,800 cycles to land at kernel start (the copy engine's
// row rate); these loads take one global round trip.
template <int BN, int kRW>
__device__ __forceinline__ void stem_stage_weights(uint8_t* wsm, const __nv_bfloat16* __restrict__ w,
                                                   const float* __restrict__ bias, int nout, int t,
                                                   uint64_t* ready) {
  constexpr int kT = 32 * kEpiWarps;
  constexpr int kN = (9 * BN + kT - 1) / kT;
  uint4 v[kN];
#pragma unroll
  for (int i = 0; i < kN; ++i) {
    const int e = t + i * kT;  // 16-byte row e of w: channel e / 9, tap e % 9
    v[i] = make_uint4(0u, 0u, 0u, 0u);
    if (e < 9 * BN && e / 9 < nout) v[i] = __ldg(reinterpret_cast<const uint4*>(w) + e);
  }
  for (int i = t; i < BN; i += kT) {
    const float b = (bias && i < nout) ? __ldg(bias + i) : 0.0f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(b);
    const __nv_bfloat16 lo = __float2bfloat16_rn(b - __bfloat162float(hi));
    *reinterpret_cast<uint4*>(wsm + 9 * BN * 16 + i * 16) =
        make_uint4((uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(lo) << 16), 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < kN; ++i) {
    const int e = t + i * kT;
    if (e < 9 * BN) {
      const int co = e / 9, tap = e - co * 9;
      const int q = kRW ? 3 * (tap % 3) + tap / 3 : tap;
      *reinterpret_cast<uint4*>(wsm + q * BN * 16 + co * 16) = v[i];
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
  if ((t & 31) == 0) mbar_arrive(ready);
}

template <int BN, bool kTS, int kRW>
__host__ __device__ constexpr uint32_t stem_a_off(int q) {
  using Cfg = StemCfg<BN, kTS, kRW>;
  return q == 9 ? Cfg::kPadOff
                : kRW ? (uint32_t)(q / 3) * Cfg::kSlotBytes + (uint32_t)(q % 3) * Cfg::kRowBytes
                      : (uint32_t)q * Cfg::kTapBytes;
}

template <int BN, bool kTS = false, int kRW = 0, bool kZ = false>
__global__ void __launch_bounds__(kIgemmThreads, 1)
    k_stem_fwd(const __grid_constant__ CUtensorMap tmA, const __nv_bfloat16* __restrict__ w,
               const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmZ,
               const IgemmParams p) {
  using Cfg = StemCfg<BN, kTS, kRW, kZ>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* wsm = smem + (size_t)S * Cfg::kStageBytes;  // resident weights
  uint8_t* osm = wsm + Cfg::kBBytes;                   // output staging (kTS)
  uint64_t* full = reinterpret_cast<uint64_t*>(osm + Cfg::kOutBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* wfull = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  const int num_tiles = p.num_m_tiles;
  const int HW = p.H * p.W;

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kEpiWarps);
    }
    mbar_init(drain, 1);
    mbar_init(wfull, kEpiWarps);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    if (kTS) tma_prefetch_desc(&tmY);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  if (warp >= kEpiBase) {
    // the tenth (padding) tap: ones in A channels 0-1 of every stage
    const int t = threadIdx.x - 32 * kEpiBase;
    for (int st = 0; st < S; ++st) {
      uint4* z = reinterpret_cast<uint4*>(smem + (size_t)st * Cfg::kStageBytes + Cfg::kPadOff);
      for (int i = t; i < (int)(Cfg::kTapBytes / 16); i += 32 * kEpiWarps) z[i] = make_uint4(0x3F803F80u, 0, 0, 0);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel's writes are visible from here on

  // resident weights and the bias tap, staged by the epilogue warps while the
  // producers already stream x (the MMA waits on wfull)
  if (warp >= kEpiBase)
    stem_stage_weights<BN, kRW>(wsm, w, p.bias, p.nout, threadIdx.x - 32 * kEpiBase, wfull);

  if (warp < kProd) {
    if (lane == 0) {
      // box-parallel: every producer takes every kProd-th box of each stage
      // (producer 0 posts the stage's byte count), so the first stage lands
      // after its own boxes instead of behind kProd stages' worth of boxes
      // interleaved on the copy engine.  Measured on the 64x64 stem with one
      // producer per stage: the first tile's data arrived ~4,900 cycles after
      // its boxes were issued.
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns, p.status, abort_flag)) {
            ok = false;
            break;
          }
          const int p0 = tile * BM;
          const int n0 = p0 / HW, rem = p0 - n0 * HW;
          const int h0 = rem / p.W, w0 = rem - h0 * p.W;
          uint8_t* sa = smem + (size_t)stage * Cfg::kStageBytes;
          if constexpr (kRW != 0) {
            // slot s: image rows h0 - 1 .. h0 + R, columns s - 1 .. s - 2 + W
            if (warp == 0) mbar_arrive_expect_tx(&full[stage], 3 * Cfg::kSlotBytes);
            constexpr int kRows = Cfg::kRowsPerTile + 2;
            for (int b = warp; b < 3 * kRows * Cfg::kRowParts; b += kProd) {
              const int part = b % Cfg::kRowParts, rho = (b / Cfg::kRowParts) % kRows;
              const int sh = b / (Cfg::kRowParts * kRows);
              tma_load_3d(sa + sh * Cfg::kSlotBytes + rho * Cfg::kRowBytes + part * 2 * Cfg::kBoxElems, &tmA,
                          &full[stage], (sh - 1) * 8 + part * Cfg::kBoxElems, h0 - 1 + rho, n0);
            }
          } else {
            if (warp == 0) mbar_arrive_expect_tx(&full[stage], 9 * Cfg::kTapBytes);
            for (int t = warp; t < 9; t += kProd)
              tma_load_im2col_4d(sa + t * Cfg::kTapBytes, &tmA, &full[stage], 0, w0 - 1, h0 - 1, n0,
                                 (uint16_t)(t % 3), (uint16_t)(t / 3));
          }
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        int n = issued < S ? issued : S;
        for (int i = 0; i < n; ++i) {
          if (--stage < 0) {
            stage = S - 1;
            phase ^= 1;
          }
          mbar_wait(&full[stage], phase, drain_wait_ns(p.wait_ns), nullptr, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0, 0);
      int stage = 0, buf = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = mbar_wait(wfull, 0, p.wait_ns, p.status, abort_flag);
      tc_fence_after();
      const uint32_t b_base = smem_u32(wsm);
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        if (!mbar_wait(&tempty[buf], acc_phase ^ 1, p.wait_ns, p.status, abort_flag)) break;
        if (!mbar_wait(&full[stage], phase, p.wait_ns, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + (size_t)stage * Cfg::kStageBytes);
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
#pragma unroll
        for (int j = 0; j < 5; ++j) {
          // K slots 2j, 2j + 1: the second's distance from the first is the LBO
          constexpr uint32_t kOff[10] = {stem_a_off<BN, kTS, kRW>(0), stem_a_off<BN, kTS, kRW>(1),
                                         stem_a_off<BN, kTS, kRW>(2), stem_a_off<BN, kTS, kRW>(3),
                                         stem_a_off<BN, kTS, kRW>(4), stem_a_off<BN, kTS, kRW>(5),
                                         stem_a_off<BN, kTS, kRW>(6), stem_a_off<BN, kTS, kRW>(7),
                                         stem_a_off<BN, kTS, kRW>(8), stem_a_off<BN, kTS, kRW>(9)};
          tc_mma_bf16(d_tmem, smem_desc(a_base + kOff[2 * j], kOff[2 * j + 1] - kOff[2 * j], 128, kSwizzleNone),
                      smem_desc(b_base + 2 * j * Cfg::kBTap, Cfg::kBTap, 128, kSwizzleNone), idesc,
                      j ? 1u : 0u);
        }
        tc_commit(&empty[stage]);
        tc_commit(&tfull[buf]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
        if (++buf == 2) {
          buf = 0;
          acc_phase ^= 1;
        }
      }
      tc_commit(drain);
      mbar_wait(drain, 0, p.wait_ns, nullptr, nullptr);
    }
    __syncwarp();
  } else if constexpr (kTS) {
    // epilogue, TMA-store path: warp (q, half) owns pixels 32q.. of the tile
    // and channels 64 half..; bias + activation in fp32, one bf16 rounding,
    // staged swizzled, one TMA store per tile (two with kZ: z, then y, in one
    // bulk group)
    const int q = warp & 3;
    const int half = (warp - kEpiBase) >> 2;
    const int col_off = half * 64;
    const int ew = warp - kEpiBase;
    int buf = 0, sb = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      if (!mbar_wait(&tfull[buf], acc_phase, p.wait_ns, p.status, abort_flag)) break;
      tc_fence_after();
      // the store issued from this buffer two tiles ago has read it
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
      uint8_t* stg = osm + (size_t)(ew * 2 + sb) * Cfg::kStageOutBytes + lane * 128;
      // z's boxes follow y's 2 x kEpiWarps boxes
      uint8_t* stz = osm + (size_t)(2 * kEpiWarps + ew * 2 + sb) * Cfg::kStageOutBytes + lane * 128;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + col_off);
      uint32_t v[2][32];
      tmem_ld_32x32b_x32(taddr, v[0]);
      tmem_ld_32x32b_x32(taddr + 32u, v[1]);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint4 u, uz;
          __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
          __nv_bfloat162* hz = reinterpret_cast<__nv_bfloat162*>(&uz);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float f0 = __uint_as_float(v[j][8 * g + 2 * i]);  // conv + bias
            float f1 = __uint_as_float(v[j][8 * g + 2 * i + 1]);
            if (kZ) hz[i] = __floats2bfloat162_rn(f0, f1);
            if (p.act == CONV3X3_ACT_SILU) {
              f0 = silu_tanh_f32(f0);
              f1 = silu_tanh_f32(f1);
            } else if (p.act == CONV3X3_ACT_LRELU) {
              f0 = f0 >= 0.0f ? f0 : 0.2f * f0;
              f1 = f1 >= 0.0f ? f1 : 0.2f * f1;
            }
            h[i] = __floats2bfloat162_rn(f0, f1);
          }
          const int chunk = (4 * j + g) ^ (lane & 7);
          *reinterpret_cast<uint4*>(stg + chunk * 16) = u;
          if (kZ) *reinterpret_cast<uint4*>(stz + chunk * 16) = uz;
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tempty[buf]);
        // one bulk group per tile (empty past the last pixel), so that
        // "all but the newest group" is always the store two tiles back
        const int row0 = tile * BM + q * 32;
        if (row0 < p.P && col_off < p.nout) {
          if (kZ)
            tma_store_2d(&tmZ, osm + (size_t)(2 * kEpiWarps + ew * 2 + sb) * Cfg::kStageOutBytes, col_off,
                         row0);
          tma_store_2d(&tmY, osm + (size_t)(ew * 2 + sb) * Cfg::kStageOutBytes, col_off, row0);
        }
        bulk_commit();
      }
      sb ^= 1;
      if (++buf == 2) {
        buf = 0;
        acc_phase ^= 1;
      }
    }
    // every store has read its staging buffer before the CTA's shared memory
    // goes away (the writes themselves complete with the grid)
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  } else {
    // epilogue: as in k_igemm with one 128-pixel sub-tile (the two warps of a
    // lane quarter take half the columns each); the bias is in the accumulator
    constexpr int kCols = BN / 2;
    IgemmParams pe = p;
    pe.bias = nullptr;
    const int q = warp & 3;
    const int half = (warp - kEpiBase) >> 2;
    const int col_off = half * kCols;
    const int row = q * 32 + lane;
    int buf = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      if (!mbar_wait(&tfull[buf], acc_phase, p.wait_ns, p.status, abort_flag)) break;
      tc_fence_after();
      const long long pix = (long long)tile * BM + row;
      const bool valid = pix < p.P;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + col_off);
#pragma unroll 1
      for (int j = 0; j < kCols / 32; ++j) {
        const int col0 = col_off + j * 32;
        const bool live = valid && col0 < p.nout;
        // the accumulator already holds conv + bias (the padding tap)
        const float bv[32] = {};
        const uint4 zr[4] = {};
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + (uint32_t)(j * 32), v);
        tmem_ld_wait();
        if (live) store_chunk<true, 0, true>(pe, pix, col0, v, bv, zr);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      if (++buf == 2) {
        buf = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, Cfg::kTmemCols);
}

// ----------------------------------------------------------------------------
// input gradient with 8 output channels (the stem): dy's 3x3 window folded in
// after a single pass over dy
// ----------------------------------------------------------------------------
// dx[h][w][c] = sum_{r,s} T[h + 1 - r][w + 1 - s][(3 r + s) * 8 + c], where
// T = dy x Wt is a plain GEMM over dy's K channels: Wt[(3 r + s) * 8 + c][k] =
// w[k][r][s][c], 72 columns (padded to N = 80).  A CTA tile is R = 128 / W
// rows of dx of one image; the tensor cores produce T for the R + 2 dy rows
// around them (one TMA box per 64 channels: rows above the image or below it
// read as zero), the epilogue warps stage T in shared memory and sum the nine
// shifted slices.  dy is read about (R + 2) / R times instead of nine times.
constexpr int kSdEpiWarps = 8;
constexpr int kSdThreads = 32 * (kProd + 1 + kSdEpiWarps);
constexpr int kSdN = 80;                  // MMA N: 72 used columns of T
// floats per staged T row (72 used): a pitch of 76 words puts the float4
// stores of eight consecutive T pixels on eight distinct 4-bank groups, where
// 72 (8 banks apart) wrote two pixels per group; the gather's reads stay
// spread evenly.  Measured on the 64x64 stem: staging a tile's T took ~1300
// cycles at pitch 72.
constexpr int kSdTPitch = 76;
constexpr uint32_t kSdChunkBytes = 256u * 128u;  // room for 256 dy pixels x 64 channels
constexpr int kSdStages = 2;

struct StemDgradParams {
  void* out;
  int out_f32;
  const __nv_bfloat16* zin;  // optional act'(z_in) scaling (laid out like dx)
  int zin_act;
  int P, H, W, K, R;         // dx pixels, image height / width, dy channels, dx rows per tile
  int num_tiles;
  unsigned* status;
  unsigned long long wait_ns;
};

__host__ __device__ constexpr size_t stem_dgrad_smem(int K) {
  return (size_t)kSdStages * (K / 64) * kSdChunkBytes  // dy stages
         + (size_t)(K / 8) * kSdN * 16                   // Wt, no-swizzle K-major
         + (size_t)256 * kSdTPitch * 4                   // staged T
         + 1024 + 256;                                   // alignment, barriers
}
static_assert(stem_dgrad_smem(128) <= 227 * 1024, "shared memory per CTA at 128 dy channels");

__global__ void __launch_bounds__(kSdThreads, 1)
    k_stem_dgrad(const __grid_constant__ CUtensorMap tmDY, const __nv_bfloat16* __restrict__ w,
                 const StemDgradParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int kchunks = p.K / 64;
  const uint32_t stage_bytes = (uint32_t)kchunks * kSdChunkBytes;
  uint8_t* wsm = smem + (size_t)kSdStages * stage_bytes;
  const uint32_t wgroup_bytes = kSdN * 16;  // one 8-channel K group of Wt: 80 rows x 16 B
  float* tsm = reinterpret_cast<float*>(wsm + (size_t)(p.K / 8) * wgroup_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(tsm + 256 * kSdTPitch);
  uint64_t* empty = full + kSdStages;
  uint64_t* tfull = empty + kSdStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* tready = tempty + 2;  // every epilogue warp has staged its T rows
  uint64_t* tdone = tready + 1;   // every epilogue warp has finished reading them
  uint64_t* drain = tdone + 1;
  uint64_t* wready = drain + 1;   // Wt is staged
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wready + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  const int rows_per_img = p.H / p.R;
  const int tpix = (p.R + 2) * p.W;  // T pixels of a tile (<= 256)

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < kSdStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kSdEpiWarps);
    }
    mbar_init(tready, kSdEpiWarps);
    mbar_init(tdone, kSdEpiWarps);
    mbar_init(drain, 1);
    mbar_init(wready, kSdThreads / 32 - 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmDY);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel's writes are visible from here on

  // Every warp but the producer stages Wt from w [K][3][3][8] while dy already
  // streams in: element (n = 8 t + c, k) at group k / 8, row n, byte 2 (k % 8);
  // rows 72..79 are zero.  One 16-byte load per (k, 8 consecutive n).  Staged
  // before the copies by the whole CTA with 2-byte loads, it held the first dy
  // box back ~3,700 cycles.
  if (warp != 0) {
    const int t = threadIdx.x - 32, nt = kSdThreads - 32;
    for (int e = t; e < p.K * 9; e += nt) {
      const int k = e / 9, n8 = e - k * 9;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(w + (size_t)k * 72) + n8);
      const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&v);
      uint8_t* dst = wsm + (size_t)(k >> 3) * wgroup_bytes + (size_t)(8 * n8) * 16 + 2 * (k & 7);
#pragma unroll
      for (int i = 0; i < 8; ++i) *reinterpret_cast<__nv_bfloat16*>(dst + i * 16) = h[i];
    }
    for (int e = t; e < (p.K / 8) * (kSdN - 72); e += nt) {
      const int g = e / (kSdN - 72), n = 72 + e - g * (kSdN - 72);
      *reinterpret_cast<uint4*>(wsm + (size_t)g * wgroup_bytes + n * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(wready);
  }

  if (warp < kProd) {
    // ------------------------------------------------------------ TMA producer (warp 0)
    if (warp == 0 && lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint32_t box_bytes = (uint32_t)tpix * 128u;
      for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
        if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns, p.status, abort_flag)) {
          ok = false;
          break;
        }
        const int n0 = tile / rows_per_img, h0 = (tile - n0 * rows_per_img) * p.R;
        uint8_t* sa = smem + (size_t)stage * stage_bytes;
        mbar_arrive_expect_tx(&full[stage], (uint32_t)kchunks * box_bytes);
        for (int c = 0; c < kchunks; ++c)
          tma_load_4d(sa + (size_t)c * kSdChunkBytes, &tmDY, &full[stage], c * 64, 0, h0 - 1, n0);
        ++issued;
        if (++stage == kSdStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        int n = issued < kSdStages ? issued : kSdStages;
        for (int i = 0; i < n; ++i) {
          if (--stage < 0) {
            stage = kSdStages - 1;
            phase ^= 1;
          }
          mbar_wait(&full[stage], phase, drain_wait_ns(p.wait_ns), nullptr, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, kSdN, 0, 0);
      const uint32_t sbase = smem_u32(smem), wbase = smem_u32(wsm);
      int stage = 0, buf = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = mbar_wait(wready, 0, p.wait_ns, p.status, abort_flag);
      for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
        if (!mbar_wait(&tempty[buf], acc_phase ^ 1, p.wait_ns, p.status, abort_flag)) break;
        if (!mbar_wait(&full[stage], phase, p.wait_ns, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t a0 = sbase + (uint32_t)stage * stage_bytes;
        const uint32_t d0 = tmem_base + (uint32_t)(buf * 2 * kSdN);
        for (int c = 0; c < kchunks; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // A: 128 dy pixels x 16 channels (SW128 K-major); B: 16 channels of Wt
            // (no swizzle, K groups 1280 bytes apart, 8-row groups 128 bytes apart)
            const uint64_t bdesc =
                smem_desc(wbase + (uint32_t)((c * 4 + kk) * 2) * (kSdN * 16), kSdN * 16, 128, kSwizzleNone);
#pragma unroll
            for (int u = 0; u < 2; ++u)
              tc_mma_bf16(d0 + (uint32_t)(u * kSdN),
                          smem_desc(a0 + (uint32_t)c * kSdChunkBytes + (uint32_t)u * 16384u + kk * 32, 16,
                                    1024, kSwizzle128B),
                          bdesc, idesc, (c | kk) != 0 ? 1u : 0u);
          }
        tc_commit(&empty[stage]);
        tc_commit(&tfull[buf]);
        if (++stage == kSdStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++buf == 2) {
          buf = 0;
          acc_phase ^= 1;
        }
      }
      tc_commit(drain);
      mbar_wait(drain, 0, p.wait_ns, nullptr, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // warp (q = lane quarter, u = half): T pixel u*128 + 32 q + lane, staged in
    // shared memory; then every thread sums four channels of one dx pixel.
    const int ew = warp - (kProd + 1);
    const int q = warp & 3, u = ew >> 2;
    const int tp = u * 128 + q * 32 + lane;
    const int e = ew * 32 + lane;  // 0..255
    const int o = e >> 1, ch = (e & 1) * 4;
    const int orow = o / p.W, ocol = o - orow * p.W;
    int buf = 0;
    uint32_t acc_phase = 0, tph = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      if (!mbar_wait(&tfull[buf], acc_phase, p.wait_ns, p.status, abort_flag)) break;
      // the previous tile's gather must be done before T is overwritten
      if (!mbar_wait(tdone, tph ^ 1, p.wait_ns, p.status, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * 2 * kSdN + u * kSdN);
      uint32_t v0[32], v1[32], v2[32];
      tmem_ld_32x32b_x32(taddr, v0);
      tmem_ld_32x32b_x32(taddr + 32, v1);
      tmem_ld_32x32b_x32(taddr + 48, v2);  // columns 48..79 (72..79 unused)
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      if (tp < tpix) {
        float4* trow = reinterpret_cast<float4*>(tsm + (size_t)tp * kSdTPitch);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          trow[i] = make_float4(__uint_as_float(v0[4 * i]), __uint_as_float(v0[4 * i + 1]),
                                __uint_as_float(v0[4 * i + 2]), __uint_as_float(v0[4 * i + 3]));
#pragma unroll
        for (int i = 0; i < 8; ++i)
          trow[8 + i] = make_float4(__uint_as_float(v1[4 * i]), __uint_as_float(v1[4 * i + 1]),
                                    __uint_as_float(v1[4 * i + 2]), __uint_as_float(v1[4 * i + 3]));
        // columns 64..71 = v2[16..23]
        trow[16] = make_float4(__uint_as_float(v2[16]), __uint_as_float(v2[17]), __uint_as_float(v2[18]),
                               __uint_as_float(v2[19]));
        trow[17] = make_float4(__uint_as_float(v2[20]), __uint_as_float(v2[21]), __uint_as_float(v2[22]),
                               __uint_as_float(v2[23]));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(tready);
      if (!mbar_wait(tready, tph, p.wait_ns, p.status, abort_flag)) break;
      // gather: dx(orow, ocol) channels ch..ch+3
      const int n0 = tile / rows_per_img, h0 = (tile - n0 * rows_per_img) * p.R;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < 3; ++r)
#pragma unroll
        for (int s = 0; s < 3; ++s) {
          const int wc = ocol + 1 - s;
          if (wc >= 0 && wc < p.W) {
            const float4 t = *reinterpret_cast<const float4*>(
                tsm + (size_t)((orow + 2 - r) * p.W + wc) * kSdTPitch + (r * 3 + s) * 8 + ch);
            acc[0] += t.x;
            acc[1] += t.y;
            acc[2] += t.z;
            acc[3] += t.w;
          }
        }
      const long long pix = ((long long)n0 * p.H + h0 + orow) * p.W + ocol;
      if (p.zin) {
        const uint2 zz = *reinterpret_cast<const uint2*>(p.zin + pix * 8 + ch);
        const __nv_bfloat162* zh = reinterpret_cast<const __nv_bfloat162*>(&zz);
        const float2 z0 = __bfloat1622float2(zh[0]), z1 = __bfloat1622float2(zh[1]);
        acc[0] *= act_grad_f32(p.zin_act, z0.x);
        acc[1] *= act_grad_f32(p.zin_act, z0.y);
        acc[2] *= act_grad_f32(p.zin_act, z1.x);
        acc[3] *= act_grad_f32(p.zin_act, z1.y);
      }
      if (p.out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(p.out) + pix * 8 + ch) =
            make_float4(acc[0], acc[1], acc[2], acc[3]);
      } else {
        uint2 o2;
        __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o2);
        oh[0] = __floats2bfloat162_rn(acc[0], acc[1]);
        oh[1] = __floats2bfloat162_rn(acc[2], acc[3]);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + pix * 8 + ch) = o2;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(tdone);
      tph ^= 1;
      if (++buf == 2) {
        buf = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, 512);
}

// ----------------------------------------------------------------------------
// input gradient with 8 output channels, image width 64: row bands
// ----------------------------------------------------------------------------
// The same T = dy x Wt formulation as k_stem_dgrad, but each CTA owns a band of
// consecutive image rows (rows of all images in one sequence, n * H + h) and
// forms T once per dy row: chunks of two dy rows (128 pixels, one M = 128 MMA
// per 16 channels) stream through four stages, the epilogue stages each
// chunk's two T rows in a ring of four T rows in shared memory, and dx row r is
// summed as soon as T rows r - 1 .. r + 1 are staged (T rows of another image,
// or outside the batch, count as zero).  dy crosses the copy engine and the
// tensor cores about once (plus two halo rows per band) instead of twice.
constexpr int kSrW = 64;                             // image width
constexpr int kSrTPitch = 76;                        // floats per staged T pixel (72 used)
constexpr uint32_t kSrTRow = kSrW * kSrTPitch * 4;   // one staged T row
constexpr int kSrRing = 4;                           // staged T rows
constexpr int kSrStages = 4;
constexpr uint32_t kSrChunkBytes = 2u * kSrW * 128u;  // two dy rows x 64 channels
static_assert(kSrTPitch % 4 == 0, "T pixels must stay 16-byte aligned");

struct StemDgradRowsParams {
  void* out;
  int out_f32;
  const __nv_bfloat16* zin;  // optional act'(z_in) scaling (laid out like dx)
  int zin_act;
  int NH, H, K;              // image rows of the batch, rows per image, dy channels
  int band;                  // dx rows per CTA
  unsigned* status;
  unsigned long long wait_ns;
};

__host__ __device__ constexpr size_t stem_dgrad_rows_smem(int K) {
  return (size_t)kSrStages * (K / 64) * kSrChunkBytes  // dy stages
         + (size_t)(K / 8) * kSdN * 16                   // Wt, no-swizzle K-major
         + (size_t)kSrRing * kSrTRow                     // staged T rows
         + 1024 + 256;                                   // alignment, barriers
}

__global__ void __launch_bounds__(kSdThreads, 1)
    k_stem_dgrad_rows(const __grid_constant__ CUtensorMap tmDY, const __nv_bfloat16* __restrict__ w,
                      const StemDgradRowsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int kchunks = p.K / 64;
  const uint32_t stage_bytes = (uint32_t)kchunks * kSrChunkBytes;
  uint8_t* wsm = smem + (size_t)kSrStages * stage_bytes;
  const uint32_t wgroup_bytes = kSdN * 16;  // one 8-channel K group of Wt: 80 rows x 16 B
  uint8_t* ring = wsm + (size_t)(p.K / 8) * wgroup_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)kSrRing * kSrTRow);
  uint64_t* empty = full + kSrStages;
  uint64_t* tfull = empty + kSrStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* tready = tempty + 2;  // every epilogue warp has staged its part of a chunk
  uint64_t* tdone = tready + 1;   // every epilogue warp has finished the gather after it
  uint64_t* drain = tdone + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  // this CTA's dx rows [g0, g1) and the T rows [t0, t1) they read
  const int g0 = blockIdx.x * p.band;
  const int g1 = min(p.NH, g0 + p.band);
  const int t0 = max(g0 - 1, 0), t1 = min(g1 + 1, p.NH);
  const int nchunks = (t1 - t0 + 1) / 2;

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < kSrStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kSdEpiWarps);
    }
    mbar_init(tready, kSdEpiWarps);
    mbar_init(tdone, kSdEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmDY);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  pdl_wait();  // w is read below
  // Wt from w [K][3][3][8]: element (n = 8 t + c, k) at group k/8, row n, 2 (k % 8) bytes;
  // rows 72..79 are zero
  for (int e = threadIdx.x; e < (p.K / 8) * kSdN; e += kSdThreads) {
    const int g = e / kSdN, n = e - g * kSdN;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < 72) {
      __nv_bfloat16 h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = w[(size_t)(g * 8 + i) * 72 + n];
      v = *reinterpret_cast<const uint4*>(h);
    }
    *reinterpret_cast<uint4*>(wsm + (size_t)g * wgroup_bytes + n * 16) = v;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < kProd) {
    // ------------------------------------------------------------ TMA producer (warp 0)
    if (warp == 0 && lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int j = 0; j < nchunks && ok; ++j) {
        if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns, p.status, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + (size_t)stage * stage_bytes;
        mbar_arrive_expect_tx(&full[stage], stage_bytes);
        for (int c = 0; c < kchunks; ++c)  // rows past the batch read as zero
          tma_load_3d(sa + (size_t)c * kSrChunkBytes, &tmDY, &full[stage], c * 64, 0, t0 + 2 * j);
        ++issued;
        if (++stage == kSrStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        int n = issued < kSrStages ? issued : kSrStages;
        for (int i = 0; i < n; ++i) {
          if (--stage < 0) {
            stage = kSrStages - 1;
            phase ^= 1;
          }
          mbar_wait(&full[stage], phase, drain_wait_ns(p.wait_ns), nullptr, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, kSdN, 0, 0);
      const uint32_t sbase = smem_u32(smem), wbase = smem_u32(wsm);
      int stage = 0, buf = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int j = 0; j < nchunks && ok; ++j) {
        if (!mbar_wait(&tempty[buf], acc_phase ^ 1, p.wait_ns, p.status, abort_flag)) break;
        if (!mbar_wait(&full[stage], phase, p.wait_ns, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t a0 = sbase + (uint32_t)stage * stage_bytes;
        const uint32_t d0 = tmem_base + (uint32_t)(buf * 128);
        for (int c = 0; c < kchunks; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            // A: 128 dy pixels x 16 channels (SW128 K-major); B: 16 channels of Wt
            tc_mma_bf16(d0, smem_desc(a0 + (uint32_t)c * kSrChunkBytes + kk * 32, 16, 1024, kSwizzle128B),
                        smem_desc(wbase + (uint32_t)((c * 4 + kk) * 2) * (kSdN * 16), kSdN * 16, 128,
                                  kSwizzleNone),
                        idesc, (c | kk) != 0 ? 1u : 0u);
        tc_commit(&empty[stage]);
        tc_commit(&tfull[buf]);
        if (++stage == kSrStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++buf == 2) {
          buf = 0;
          acc_phase ^= 1;
        }
      }
      tc_commit(drain);
      mbar_wait(drain, 0, p.wait_ns, nullptr, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // warp (q = lane quarter, h = half): T pixel 32 q + lane of the chunk;
    // half 0 stages columns 0..31 and 64..71, half 1 columns 32..63
    const int ew = warp - (kProd + 1);
    const int q = warp & 3, h = ew >> 2;
    const int tp = q * 32 + lane;  // pixel of the chunk: row tp / 64, column tp % 64
    const int et = ew * 32 + lane;  // 0..255: gather thread
    const int gpx = et >> 2, gc = (et & 3) * 2;  // gather: pixel, channel pair
    int buf = 0;
    uint32_t acc_phase = 0, tph = 0;
    int next = g0;  // next dx row to sum
    bool ok = true;
    for (int j = 0; j <= nchunks && ok; ++j) {
      const bool staging = j < nchunks;
      // the previous gather has read the ring slots this chunk overwrites
      if (!mbar_wait(tdone, tph ^ 1, p.wait_ns, p.status, abort_flag)) break;
      if (staging) {
        if (!mbar_wait(&tfull[buf], acc_phase, p.wait_ns, p.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * 128);
        uint32_t v[32], v8[8];
        tmem_ld_32x32b_x32(taddr + (h ? 32u : 0u), v);
        if (h == 0) tmem_ld_32x32b_x8(taddr + 64u, v8);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        const int slot = (2 * j + (tp >> 6)) & (kSrRing - 1);
        float4* trow = reinterpret_cast<float4*>(ring + (size_t)slot * kSrTRow + (size_t)(tp & 63) * kSrTPitch * 4);
        const int c4 = h ? 8 : 0;  // first float4 of this warp's 32 columns
#pragma unroll
        for (int i = 0; i < 8; ++i)
          trow[c4 + i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                     __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        if (h == 0) {
          trow[16] = make_float4(__uint_as_float(v8[0]), __uint_as_float(v8[1]), __uint_as_float(v8[2]),
                                 __uint_as_float(v8[3]));
          trow[17] = make_float4(__uint_as_float(v8[4]), __uint_as_float(v8[5]), __uint_as_float(v8[6]),
                                 __uint_as_float(v8[7]));
        }
        if (++buf == 2) {
          buf = 0;
          acc_phase ^= 1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(tready);
      if (!mbar_wait(tready, tph, p.wait_ns, p.status, abort_flag)) {
        ok = false;
        break;
      }
      // T rows t0 .. t0 + 2 j + 1 are staged: sum every dx row r whose T rows
      // r - 1 .. r + 1 are (after the last chunk: every remaining row -- the
      // rows past the staged ones are past the batch and read as zero)
      const int hi = staging ? t0 + 2 * j : p.NH;
      for (; next < g1 && next <= hi; ++next) {
        const int r = next, img = r / p.H;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int rk = 0; rk < 3; ++rk) {
          const int tr = r + 1 - rk;  // T row
          if (tr < 0 || tr >= p.NH || tr / p.H != img) continue;
          const float* tb = reinterpret_cast<const float*>(ring + (size_t)((tr - t0) & (kSrRing - 1)) * kSrTRow);
#pragma unroll
          for (int s = 0; s < 3; ++s) {
            const int px = gpx + 1 - s;
            if (px < 0 || px >= kSrW) continue;
            const float2 t = *reinterpret_cast<const float2*>(tb + px * kSrTPitch + (rk * 3 + s) * 8 + gc);
            a0 += t.x;
            a1 += t.y;
          }
        }
        const long long pix = (long long)r * kSrW + gpx;
        if (p.zin) {
          const float2 z = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p.zin + pix * 8 + gc));
          a0 *= act_grad_f32(p.zin_act, z.x);
          a1 *= act_grad_f32(p.zin_act, z.y);
        }
        if (p.out_f32)
          *reinterpret_cast<float2*>(static_cast<float*>(p.out) + pix * 8 + gc) = make_float2(a0, a1);
        else
          *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + pix * 8 + gc) =
              __floats2bfloat162_rn(a0, a1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(tdone);
      tph ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, 256);
}

// ----------------------------------------------------------------------------
// wgrad split-K implicit GEMM
// ----------------------------------------------------------------------------
constexpr int kWgTaps = 3;                       // taps per CTA tile (one kernel row)
constexpr int kWgPix = 64;                       // pixels per k-block
constexpr uint32_t kWgABytes = 128 * kWgPix * 2;  // dy: 64 px x 128 Cout
constexpr uint32_t kWgBBytes = 128 * kWgPix * 2;  // x: 64 px x 128 Cin, per tap
constexpr uint32_t kWgOnesBytes = 8192;          // 64 px x 64 columns of bf16 ones
constexpr int kWgTmemCols = 512;                 // 3 x 128 dw columns + 16 dbias columns (384..399)
constexpr int kWgBiasCol = kWgTaps * 128;
static_assert(!kWgStageParallel, "the wgrad stages are shared box-parallel by the producers");

// Stage layout of k_wgrad.  kHW = 0 (im2col x): dy (two 64-pixel x 64-channel
// boxes), then per tap two 64-pixel x 64-channel im2col boxes of x, then the
// ones block.  kHW = image width 16, 32 or 64 (row-shifted x): a k-block is
// R = 64 / kHW whole image rows; per 64-channel half j and image row i one
// tiled box holds x[h][-1 .. kHW][64 channels] (the columns outside the image
// read zero), in a slot of kSlot bytes, slots ordered [j][i]; tap s of the
// kernel row reads that box from row s on, so one box serves all three taps.
// Slot half j = 2 is all ones (the dbias block, at the same offsets).
template <int kHW>
struct WgCfg {
  static constexpr int R = kHW ? kWgPix / kHW : 0;
  static constexpr uint32_t kSlot = kHW ? (uint32_t)((kHW + 2) * 128 + 1023) / 1024 * 1024 : 0;
  static constexpr uint32_t kXBytes = kHW ? 3u * R * kSlot : kWgTaps * kWgBBytes + kWgOnesBytes;
  static constexpr uint32_t kStageBytes = kWgABytes + kXBytes;
  static constexpr int kStagesFit = (int)((220u * 1024u) / kStageBytes);
  static constexpr int kStages = kStagesFit > 6 ? 6 : kStagesFit;
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + 256 + 1024 + 8 * 1024;
  static_assert(kHW == 0 || kHW == 16 || kHW == 32 || kHW == 64, "row-shifted x for widths 16, 32, 64");
  static_assert(kStages >= 3, "wgrad stage ring too shallow");
  static_assert(kStageBytes % 1024 == 0 && kSlot % 1024 == 0, "swizzle atoms must stay 1 KB aligned");
  static_assert(kStages * kStageBytes >= 2 * kWgEpiWarps * 4 * 4096, "partial staging fits in the stage ring");
};

struct WgradParams {
  float* part;  // [S][Cout][9*Cin] then [S][Cout]
  int P, H, W, Cin, Cout;
  int ca;       // channel-split input: channels [0, ca) from tmX, [ca, Cin) from tmX2 (ca % 64 == 0)
  int ustride;  // conv stride: output pixel (h, w) reads x around (u*h, u*w); P, H, W are dy's grid
  int kb_total, kb_per_split, S;
  int num_mb, num_cb;  // 128-wide blocks of Cout and Cin
  unsigned* status;
  unsigned long long wait_ns;
  int part_tma = 0;    // the dw partials leave through tmPart (see wg_store_partials)
  int mb0 = 0;         // first 128-channel block of Cout this launch covers (k_wgrad)
};

// The dw partials of one wgrad CTA tile -- TMEM lanes = 128 output channels
// from k0, columns 128 t + c = tap 3 tr + t, input channel cb * 128 + c (tap
// 2's columns 64.. sit `gap` columns later in the pair tile that owns dbias)
// -- written to part [S][Cout][9][Cin] through TMA tensor stores.  The
// twelve 32-column chunks n = 4 t + j of lane quarter q are shared by two
// warps (the epilogue warp takes n0 .. n1 = 0 .. 6, the idle producer warp of
// the same quarter 6 .. 12).  A warp stages its 32 rows of a chunk (4 KB,
// 128-byte swizzle) in four rotating buffers of its slot of the (idle) stage
// memory at `stg`, and lane 0 stores the box {32 channels, 1 tap, 32 rows, 1
// split} of map tmPart ([S][Cout][9][Cin] fp32; rows past Cout and channels
// past Cin are clipped).  Each thread storing its own row with 16-byte stores
// made every warp store touch 32 lines: the partials then took ~19,000 cycles
// of a 73,000-cycle CTA on the 384-channel 16x16 layer.
__device__ __forceinline__ void wg_store_partials(const CUtensorMap* tmPart, uint8_t* stg, uint32_t lane_addr,
                                                  int tr, int cb, int k0, int split, int Cin, int Cout,
                                                  int q, int lane, uint32_t gap, int n0, int n1, int slot) {
  uint8_t* wbuf = stg + (size_t)slot * 4 * 4096;
#pragma unroll 1
  for (int n = n0; n < n1; ++n) {
    const int t = n >> 2, j = n & 3;
    {
      uint32_t v[32];
      tmem_ld_32x32b_x32(lane_addr + (uint32_t)(t * 128 + j * 32) + (t == 2 && j >= 2 ? gap : 0u), v);
      tmem_ld_wait();
      uint8_t* buf = wbuf + ((n - n0) & 3) * 4096;
      // the store issued from this buffer four chunks ago has read it
      if (n - n0 >= 4 && lane == 0) bulk_wait_read<3>();
      __syncwarp();
#pragma unroll
      for (int g = 0; g < 8; ++g)
        *reinterpret_cast<uint4*>(buf + lane * 128 + ((g ^ (lane & 7)) << 4)) =
            make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int c0 = cb * 128 + j * 32, r0 = k0 + q * 32;
        if (c0 < Cin && r0 < Cout) tma_store_4d(tmPart, buf, c0, tr * 3 + t, r0, split);
        bulk_commit();  // one group per chunk, empty or not
      }
    }
  }
  if (lane == 0) bulk_wait_read<0>();  // the stores' writes complete with the grid
  __syncwarp();
}

template <int kHW>
__global__ void __launch_bounds__(kThreads, 1)
    k_wgrad(const __grid_constant__ CUtensorMap tmDY, const __grid_constant__ CUtensorMap tmX,
            const __grid_constant__ CUtensorMap tmX2, const __grid_constant__ CUtensorMap tmPart,
            const WgradParams p) {
  using Cfg = WgCfg<kHW>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * Cfg::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // no early trigger: the dependent is the partials' reduction, whose blocks
  // would otherwise sit on the SMs (waiting) while this kernel runs
  const int num_tiles = p.num_mb * 3 * p.num_cb;
  const int tile = blockIdx.x % num_tiles;
  const int split = blockIdx.x / num_tiles;
  const int mb = p.mb0 + tile % p.num_mb;
  const int rest = tile / p.num_mb;
  const int cb = rest % p.num_cb;
  const int tr = rest / p.num_cb;  // kernel row r: taps 3r .. 3r+2
  const bool do_bias = (tr == 0 && cb == 0);
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
  const int HW = p.H * p.W;

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], kProd);
      mbar_init(&empty[i], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmDY);
    tma_prefetch_desc(&tmX);
    if (p.ca < p.Cin) tma_prefetch_desc(&tmX2);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kWgTmemCols);
    tmem_relinquish();
  }
  if (warp >= kEpiBase && do_bias) {  // fill every stage's ones block (bf16 1.0 = 0x3F80)
    constexpr uint32_t kOnesOff = kHW ? kWgABytes + 2u * Cfg::R * Cfg::kSlot : kWgABytes + kWgTaps * kWgBBytes;
    constexpr uint32_t kOnes = kHW ? Cfg::R * Cfg::kSlot : kWgOnesBytes;
    for (int st = 0; st < S; ++st) {
      uint4* o = reinterpret_cast<uint4*>(smem + (size_t)st * Cfg::kStageBytes + kOnesOff);
      for (int i = threadIdx.x - 32 * kEpiBase; i < (int)(kOnes / 16); i += 32 * kWgEpiWarps)
        o[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel's writes are visible from here on

  if (warp < kProd) {
    // Boxes per stage: two dy boxes (64 pixels x 64 output channels), then x:
    // im2col, per tap two 64-pixel x 64-channel boxes; row-shifted, per
    // channel half and image row one (kHW + 2)-pixel box.  Producer `warp`
    // issues boxes warp, warp + 4, ...
    if (lane == 0) {
      constexpr int kXBoxes = kHW ? 2 * Cfg::R : 2 * kWgTaps;
      constexpr uint32_t kXBox = kHW ? (uint32_t)(kHW + 2) * 128u : 8192u;
      uint32_t bytes = 0;
      for (int b = warp; b < 2 + kXBoxes; b += kProd) bytes += b < 2 ? 8192u : kXBox;
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns, p.status, abort_flag)) {
          ok = false;
          break;
        }
        const int pk = kb * kWgPix;
        const int n0 = pk / HW, rem = pk - n0 * HW;
        const int h0 = rem / p.W, w0 = rem - h0 * p.W;
        uint8_t* sa = smem + (size_t)stage * Cfg::kStageBytes;
        uint8_t* sb = sa + kWgABytes;
        mbar_arrive_expect_tx(&full[stage], bytes);
        for (int b = warp; b < 2 + kXBoxes; b += kProd) {
          if (b < 2) {
            tma_load_2d(sa + b * 8192, &tmDY, &full[stage], mb * 128 + b * 64, pk);
          } else if constexpr (kHW != 0) {
            const int j = (b - 2) / Cfg::R, i = (b - 2) - j * Cfg::R;
            const int c = cb * 128 + j * 64;  // a 64-channel box lies in one part
            const bool second = c >= p.ca;
            tma_load_4d(sb + (size_t)(j * Cfg::R + i) * Cfg::kSlot, second ? &tmX2 : &tmX, &full[stage],
                        second ? c - p.ca : c, -1, h0 + i + tr - 1, n0);
          } else {
            const int t = (b - 2) >> 1, j = (b - 2) & 1;
            const int c = cb * 128 + j * 64;
            const bool second = c >= p.ca;
            tma_load_im2col_4d(sb + (t * 2 + j) * 8192, second ? &tmX2 : &tmX, &full[stage],
                               second ? c - p.ca : c, p.ustride * w0 - 1, p.ustride * h0 - 1, n0,
                               (uint16_t)t, (uint16_t)tr);
          }
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        int n = issued < S ? issued : S;
        int st = stage;
        uint32_t ph = phase;
        for (int i = 0; i < n; ++i) {
          if (--st < 0) {
            st = S - 1;
            ph ^= 1;
          }
          mbar_wait(&full[st], ph, drain_wait_ns(p.wait_ns), nullptr, nullptr);
        }
      }
    }
    __syncwarp();
    // this lane quarter's partial chunks 6 .. 11 (see wg_store_partials)
    if (p.part_tma && mbar_wait(tfull, 0, p.wait_ns, p.status, abort_flag)) {
      tc_fence_after();
      wg_store_partials(&tmPart, smem, tmem_base + ((uint32_t)(warp * 32) << 16), tr, cb, mb * 128, split, p.Cin,
                        p.Cout, warp, lane, 0u, 6, 12, kWgEpiWarps + warp);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc256 = idesc_bf16_f32(128, 256, 1, 1);
      constexpr uint32_t idesc128 = idesc_bf16_f32(128, 128, 1, 1);
      constexpr uint32_t idesc144 = idesc_bf16_f32(128, 144, 1, 1);
      const uint32_t idesc_t2 = do_bias ? idesc144 : idesc128;
      // descriptors built once; stages and K steps move the start address only
      const uint32_t sbase = smem_u32(smem);
      const uint64_t a_desc0 = smem_desc(sbase, 8192, 1024, kSwizzle128B);
      // row-shifted x: slot rows of stage 0 (addresses stay below 2^18, so
      // adding offsets >> 4 to the start field never carries out of it)
      const uint64_t x_desc0 = smem_desc(sbase + kWgABytes, Cfg::R * Cfg::kSlot, 1024, kSwizzle128B);
      constexpr uint32_t kStageStep = Cfg::kStageBytes >> 4;
      constexpr uint32_t kKStep = 2048u >> 4;
      int stage = 0;
      uint32_t phase = 0, stage_off = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full[stage], phase, p.wait_ns, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = a_desc0 + stage_off;
        const uint32_t acc0 = kb != kb0 ? 1u : 0u;
        if constexpr (kHW) {
          // K step k covers pixels 16k .. 16k + 15 of the k-block: image row
          // i = 16k / kHW, columns w0 .. w0 + 15 with w0 = 16k mod kHW; tap s
          // reads rows w0 + s .. of slot (j, i) (the box starts at column -1),
          // the two channel halves Cfg::R slots apart.  The swizzle follows the
          // absolute shared-memory address, so a start that is s rows into a
          // 1 KB swizzle atom needs no base offset.
          const uint64_t xd = x_desc0 + stage_off;
#pragma unroll
          for (int k = 0; k < kWgPix / 16; ++k) {
            const uint32_t acc = k == 0 ? acc0 : 1u;
            constexpr int kW = kHW ? kHW : 16;  // (kHW = 0 never reaches here)
            const int i = (16 * k) / kW, w0 = (16 * k) % kW;
            const uint32_t row0 = (uint32_t)i * Cfg::kSlot + (uint32_t)w0 * 128u;
#pragma unroll
            for (int t = 0; t < kWgTaps; ++t)
              tc_mma_bf16(tmem_base + (uint32_t)(t * 128), ad + (uint64_t)(k * kKStep),
                          xd + (uint64_t)((row0 + (uint32_t)t * 128u) >> 4), t == 2 ? idesc_t2 : idesc128,
                          acc);
          }
        } else {
          const uint64_t b_desc0 = smem_desc(sbase + kWgABytes, 8192, 1024, kSwizzle128B);
          const uint64_t bd = b_desc0 + stage_off;
          constexpr uint32_t kTap2 = (2 * kWgBBytes) >> 4;
#pragma unroll
          for (int k = 0; k < kWgPix / 16; ++k) {
            const uint32_t acc = k == 0 ? acc0 : 1u;
            // taps 0 and 1: four 64-channel blocks at 8 KB stride -> one N = 256 MMA
            tc_mma_bf16(tmem_base, ad + (uint64_t)(k * kKStep), bd + (uint64_t)(k * kKStep), idesc256,
                        acc);
            // tap 2 (+ the ones block as a third 64-column block when this CTA owns dbias)
            tc_mma_bf16(tmem_base + 256, ad + (uint64_t)(k * kKStep),
                        bd + (uint64_t)(kTap2 + k * kKStep), idesc_t2, acc);
          }
        }
        tc_commit(&empty[stage]);
        stage_off += kStageStep;
        if (++stage == S) {
          stage = 0;
          stage_off = 0;
          phase ^= 1;
        }
      }
      if (ok) tc_commit(tfull);
      tc_commit(drain);
      mbar_wait(drain, 0, p.wait_ns, nullptr, nullptr);
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int k = mb * 128 + row;
    if (mbar_wait(tfull, 0, p.wait_ns, p.status, abort_flag)) {
      tc_fence_after();
      const long long dwsize = (long long)p.Cout * 9 * p.Cin;
      const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
      if (p.part_tma)
        wg_store_partials(&tmPart, smem, lane_addr, tr, cb, mb * 128, split, p.Cin, p.Cout, q, lane, 0u, 0, 6, q);
#pragma unroll 1
      for (int t = 0; t < (p.part_tma ? 0 : kWgTaps); ++t) {
        const int tap = tr * 3 + t;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(lane_addr + (uint32_t)(t * 128 + j * 32), v);
          tmem_ld_wait();
          const int c0 = cb * 128 + j * 32;
          if (k < p.Cout && c0 < p.Cin) {
            float* o = p.part + (long long)split * dwsize + ((long long)k * 9 + tap) * p.Cin + c0;
#pragma unroll
            for (int g = 0; g < 4; ++g)
              if (c0 + 8 * g < p.Cin) {
                reinterpret_cast<float4*>(o + 8 * g)[0] = make_float4(
                    __uint_as_float(v[8 * g]), __uint_as_float(v[8 * g + 1]),
                    __uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]));
                reinterpret_cast<float4*>(o + 8 * g)[1] = make_float4(
                    __uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]),
                    __uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]));
              }
          }
        }
      }
      if (do_bias) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(lane_addr + (uint32_t)kWgBiasCol, v);
        tmem_ld_wait();
        if (k < p.Cout)
          p.part[(long long)p.S * dwsize + (long long)split * p.Cout + k] = __uint_as_float(v[0]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, kWgTmemCols);
}

// ----------------------------------------------------------------------------
// wgrad on two-CTA clusters (tcgen05.mma.cta_group::2)
// ----------------------------------------------------------------------------
// A pair tile is 256 output channels (128 per CTA: the MMA's M = 256 rows, dy
// MN-major) x one kernel row (three taps) x 128 input channels, over a pixel
// range.  The pair shares the x operand, each CTA staging half of its columns:
// rank 0 tap 0 and input channels 0-63 of tap 2, rank 1 tap 1 and channels
// 64-127 of tap 2.  Per 16 pixels one M = 256, N = 256 MMA covers taps 0-1
// (accumulator columns 0-127 from rank 0's half, 128-255 from rank 1's) and
// one M = 256, N = 128 MMA tap 2 (columns 256-319 and 320-383); in the pair
// that owns dbias the tap-2 MMA is N = 144 and each half ends with 8 columns
// of the static ones block, so tap 2's second half moves to columns 328-391
// and column 320 holds dbias.  Each CTA stages 40 KB per 64-pixel k-block
// where the one-CTA tile stages 64 KB for the same accumulator work, and the
// tensor core reads half the x operand from each shared memory.
constexpr uint32_t kWpX0 = kWgABytes;                      // this CTA's tap (0 or 1), two 64-channel boxes
constexpr uint32_t kWpX2 = kWgABytes + kWgBBytes;          // this CTA's 64 channels of tap 2
constexpr uint32_t kWpOnes = kWpX2 + kWgBBytes / 2;        // ones block (follows tap 2 at one box stride)
constexpr uint32_t kWpStage = kWpOnes + kWgOnesBytes;      // 48 KB
constexpr uint32_t kWpLoadBytes = kWpOnes;                 // bytes each CTA loads per k-block
constexpr int kWpBiasCol = 256 + 64;                     // rank 0's first ones column
constexpr int kWpStages = 4;
constexpr size_t kWpSmem = (size_t)kWpStages * kWpStage + 256 + 1024 + 8 * 1024;
static_assert(kWpStages >= kProd, "stage-parallel producers need S >= kProd");
static_assert(kWpStage % 1024 == 0 && kWpX2 % 1024 == 0, "swizzle atoms must stay 1 KB aligned");
static_assert(kWpStages * kWpStage >= 2 * kWgEpiWarps * 4 * 4096, "partial staging fits in the stage ring");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_wgrad_pair(const __grid_constant__ CUtensorMap tmDY, const __grid_constant__ CUtensorMap tmX,
                 const __grid_constant__ CUtensorMap tmX2, const __grid_constant__ CUtensorMap tmPart,
                 const WgradParams p) {
  constexpr int S = kWpStages;
  extern __shared__ uint8_t smem_raw[];
  // same offsets in both CTAs: the MMAs address the peer's operands at rank 0's
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * kWpStage);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  // num_mb counts 256-channel pair blocks here
  const int num_tiles = p.num_mb * 3 * p.num_cb;
  const int pair = blockIdx.x >> 1;
  const int tile = pair % num_tiles;
  const int split = pair / num_tiles;
  const int mb = tile % p.num_mb;
  const int rest = tile / p.num_mb;
  const int cb = rest % p.num_cb;
  const int tr = rest / p.num_cb;  // kernel row r: taps 3r .. 3r+2
  const bool do_bias = (tr == 0 && cb == 0);
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
  const int HW = p.H * p.W;

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmDY);
    tma_prefetch_desc(&tmX);
    if (p.ca < p.Cin) tma_prefetch_desc(&tmX2);
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(tmem_slot, kWgTmemCols);
    tmem_relinquish_pair();
  }
  if (warp >= kEpiBase && do_bias) {  // every stage's ones block (bf16 1.0 = 0x3F80)
    for (int st = 0; st < S; ++st) {
      uint4* o = reinterpret_cast<uint4*>(smem + (size_t)st * kWpStage + kWpOnes);
      for (int i = threadIdx.x - 32 * kEpiBase; i < (int)(kWgOnesBytes / 16); i += 32 * kWgEpiWarps)
        o[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel's writes are visible from here on
  const uint32_t full0 = cluster_addr(full, 0);  // rank 0's full barriers count both CTAs' bytes

  if (warp < kProd) {
    // Whole stages in turn: producer `warp` fills the k-blocks issued % kProd
    // == warp with this CTA's dy half (two 64-channel boxes), its x tap (two
    // im2col boxes) and its 64 channels of tap 2.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (issued % kProd == warp) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns, p.status, abort_flag)) {
            ok = false;
            break;
          }
          const int pk = kb * kWgPix;
          const int n0 = pk / HW, rem = pk - n0 * HW;
          const int h0 = rem / p.W, w0 = rem - h0 * p.W;
          const int cw = p.ustride * w0 - 1, chh = p.ustride * h0 - 1;
          uint8_t* sa = smem + (size_t)stage * kWpStage;
          const uint32_t fb = full0 + (uint32_t)stage * 8u;
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * kWpLoadBytes);
          const int k0 = mb * 256 + (int)rank * 128;
          tma_load_2d_pair(sa, &tmDY, fb, k0, pk);
          tma_load_2d_pair(sa + 8192, &tmDY, fb, k0 + 64, pk);
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            // j = 0, 1: this CTA's tap, channel halves; j = 2: its half of tap 2
            const int t = j < 2 ? (int)rank : 2;
            const int c = cb * 128 + (j < 2 ? j * 64 : (int)rank * 64);  // a 64-channel box lies in one part
            const bool second = c >= p.ca;
            tma_load_im2col_4d_pair(sa + kWpX0 + j * 8192, second ? &tmX2 : &tmX, fb, second ? c - p.ca : c, cw,
                                    chh, n0, (uint16_t)t, (uint16_t)tr);
          }
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        if (rank == 0) {
          // wait (bounded) for the loads still in flight
          int n = issued < S ? issued : S;
          int st = stage;
          uint32_t ph = phase;
          for (int i = 0; i < n; ++i) {
            if (--st < 0) {
              st = S - 1;
              ph ^= 1;
            }
            mbar_wait(&full[st], ph, drain_wait_ns(p.wait_ns), nullptr, nullptr);
          }
        } else {
          // rank 1's loads complete on rank 0's barriers: give them time to land
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) __nanosleep(1000);
        }
      }
    }
    __syncwarp();
    // this lane quarter's partial chunks 6 .. 11 (see wg_store_partials)
    if (p.part_tma && mbar_wait(tfull, 0, p.wait_ns, p.status, abort_flag)) {
      tc_fence_after();
      wg_store_partials(&tmPart, smem, tmem_base + ((uint32_t)(warp * 32) << 16), tr, cb,
                        mb * 256 + (int)rank * 128, split, p.Cin, p.Cout, warp, lane, do_bias ? 8u : 0u, 6, 12,
                        kWgEpiWarps + warp);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc256 = idesc_bf16_f32(256, 256, 1, 1);
      const uint32_t idesc_t2 = idesc_bf16_f32(256, do_bias ? 144 : 128, 1, 1);
      const uint32_t sbase = smem_u32(smem);
      const uint64_t a_desc0 = smem_desc(sbase, 8192, 1024, kSwizzle128B);
      const uint64_t b01_desc0 = smem_desc(sbase + kWpX0, 8192, 1024, kSwizzle128B);
      const uint64_t b2_desc0 = smem_desc(sbase + kWpX2, 8192, 1024, kSwizzle128B);
      constexpr uint32_t kStageStep = kWpStage >> 4;
      constexpr uint32_t kKStep = 2048u >> 4;  // 16 pixels of an MN-major operand
      int stage = 0;
      uint32_t phase = 0, stage_off = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full[stage], phase, p.wait_ns, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc0 = kb != kb0 ? 1u : 0u;
#pragma unroll
        for (int k = 0; k < kWgPix / 16; ++k) {
          const uint32_t acc = k == 0 ? acc0 : 1u;
          const uint64_t off = (uint64_t)(stage_off + k * kKStep);
          tc_mma_bf16_pair(tmem_base, a_desc0 + off, b01_desc0 + off, idesc256, acc);
          tc_mma_bf16_pair(tmem_base + 256, a_desc0 + off, b2_desc0 + off, idesc_t2, acc);
        }
        tc_commit_pair_mc(&empty[stage], (uint16_t)0x3);
        stage_off += kStageStep;
        if (++stage == S) {
          stage = 0;
          stage_off = 0;
          phase ^= 1;
        }
      }
      if (ok) tc_commit_pair_mc(tfull, (uint16_t)0x3);
      // every issued MMA (which reads both CTAs' shared memory and writes both
      // TMEMs) retires before either CTA releases anything
      tc_commit_pair(drain);
      mbar_wait(drain, 0, p.wait_ns, nullptr, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // TMEM lane = this CTA's output channel; column c of tap t as described
    // above the kernel.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int k = mb * 256 + (int)rank * 128 + row;
    if (mbar_wait(tfull, 0, p.wait_ns, p.status, abort_flag)) {
      tc_fence_after();
      const long long dwsize = (long long)p.Cout * 9 * p.Cin;
      const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
      const uint32_t gap = do_bias ? 8u : 0u;  // the ones columns between tap 2's halves
      if (p.part_tma)
        wg_store_partials(&tmPart, smem, lane_addr, tr, cb, mb * 256 + (int)rank * 128, split, p.Cin, p.Cout, q,
                          lane, gap, 0, 6, q);
#pragma unroll 1
      for (int t = 0; t < (p.part_tma ? 0 : kWgTaps); ++t) {
        const int tap = tr * 3 + t;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          const uint32_t col = (uint32_t)(t * 128 + j * 32) + (t == 2 && j >= 2 ? gap : 0u);
          uint32_t v[32];
          tmem_ld_32x32b_x32(lane_addr + col, v);
          tmem_ld_wait();
          const int c0 = cb * 128 + j * 32;
          if (k < p.Cout && c0 < p.Cin) {
            float* o = p.part + (long long)split * dwsize + ((long long)k * 9 + tap) * p.Cin + c0;
#pragma unroll
            for (int g = 0; g < 4; ++g)
              if (c0 + 8 * g < p.Cin) {
                reinterpret_cast<float4*>(o + 8 * g)[0] = make_float4(
                    __uint_as_float(v[8 * g]), __uint_as_float(v[8 * g + 1]),
                    __uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]));
                reinterpret_cast<float4*>(o + 8 * g)[1] = make_float4(
                    __uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]),
                    __uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]));
              }
          }
        }
      }
      if (do_bias) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(lane_addr + (uint32_t)kWpBiasCol, v);
        tmem_ld_wait();
        if (k < p.Cout)
          p.part[(long long)p.S * dwsize + (long long)split * p.Cout + k] = __uint_as_float(v[0]);
      }
    }
  }

  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc_pair(tmem_base, kWgTmemCols);
}

// ----------------------------------------------------------------------------
// wgrad, 8 input channels (the UNet stem)
// ----------------------------------------------------------------------------
// N = all nine taps x 8 channels at once: per 64-pixel k-block, x is staged as
// nine im2col boxes of 64 pixels x 8 channels (1 KB each, no swizzle); in the
// MN-major no-swizzle operand layout each box is one 8-column block of core
// matrices (8 pixels x 16 bytes), blocks 1 KB apart.  A zero block pads N to
// 80 and two blocks of ones add 16 dbias columns: one M = 128, N = 96, K = 16
// MMA per 16 pixels covers dw and dbias.
constexpr uint32_t kWc8BlockBytes = kWgPix * 16;               // 64 px x 8 channels
constexpr uint32_t kWc8BBytes = 12 * kWc8BlockBytes;           // 9 taps, zero, 2 x ones
constexpr uint32_t kWc8StageBytes = kWgABytes + kWc8BBytes;
constexpr int kWc8Stages = 6;
constexpr size_t kWc8Smem = (size_t)kWc8Stages * kWc8StageBytes + 256 + 1024;
static_assert(kWc8StageBytes % 16 == 0, "stage offsets move descriptor start fields in 16-byte units");

__global__ void __launch_bounds__(kThreads, 1)
    k_wgrad_c8(const __grid_constant__ CUtensorMap tmDY, const __grid_constant__ CUtensorMap tmX,
               const WgradParams p) {
  constexpr int S = kWc8Stages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * kWc8StageBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // no early trigger: the dependent is the partials' reduction, whose blocks
  // would otherwise sit on the SMs (waiting) while this kernel runs
  const int mb = blockIdx.x % p.num_mb;
  const int split = blockIdx.x / p.num_mb;
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
  const int HW = p.H * p.W;

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], kProd);
      mbar_init(&empty[i], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmDY);
    tma_prefetch_desc(&tmX);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  if (warp >= kEpiBase) {  // per stage: block 9 = zeros, blocks 10-11 = bf16 ones
    const int t = threadIdx.x - 32 * kEpiBase;
    for (int st = 0; st < S; ++st) {
      uint4* b = reinterpret_cast<uint4*>(smem + (size_t)st * kWc8StageBytes + kWgABytes + 9 * kWc8BlockBytes);
      for (int i = t; i < (int)(3 * kWc8BlockBytes / 16); i += 32 * kWgEpiWarps) {
        const uint32_t v = i < (int)(kWc8BlockBytes / 16) ? 0u : 0x3F803F80u;
        b[i] = make_uint4(v, v, v, v);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel's writes are visible from here on

  if (warp < kProd) {
    // boxes per stage: dy halves 0-1 (8 KB); x taps 2-10 (1 KB im2col boxes)
    if (lane == 0) {
      constexpr int kBoxes = 11;
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      uint32_t bytes = 0;
      for (int b = warp; b < kBoxes; b += kProd) bytes += b < 2 ? 8192u : kWc8BlockBytes;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns, p.status, abort_flag)) {
          ok = false;
          break;
        }
        const int pk = kb * kWgPix;
        const int n0 = pk / HW, rem = pk - n0 * HW;
        const int h0 = rem / p.W, w0 = rem - h0 * p.W;
        uint8_t* sa = smem + (size_t)stage * kWc8StageBytes;
        uint8_t* sb = sa + kWgABytes;
        mbar_arrive_expect_tx(&full[stage], bytes);
        for (int b = warp; b < kBoxes; b += kProd) {
          if (b < 2) {
            tma_load_2d(sa + b * 8192, &tmDY, &full[stage], mb * 128 + b * 64, pk);
          } else {
            const int t = b - 2;
            tma_load_im2col_4d(sb + t * kWc8BlockBytes, &tmX, &full[stage], 0, w0 - 1, h0 - 1, n0,
                               (uint16_t)(t % 3), (uint16_t)(t / 3));
          }
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        int n = issued < S ? issued : S;
        for (int i = 0; i < n; ++i) {
          if (--stage < 0) {
            stage = S - 1;
            phase ^= 1;
          }
          mbar_wait(&full[stage], phase, drain_wait_ns(p.wait_ns), nullptr, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 96, 1, 1);
      // descriptors built once for stage 0 (addresses stay below 2^18: adding
      // offsets >> 4 to the start field never carries out of it)
      const uint32_t sbase = smem_u32(smem);
      const uint64_t a_desc0 = smem_desc(sbase, 8192, 1024, kSwizzle128B);
      const uint64_t b_desc0 = smem_desc(sbase + kWgABytes, 128, kWc8BlockBytes, kSwizzleNone);
      constexpr uint32_t kStageStep = kWc8StageBytes >> 4;
      int stage = 0;
      uint32_t phase = 0, stage_off = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full[stage], phase, p.wait_ns, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kWgPix / 16; ++k)
          tc_mma_bf16(tmem_base, a_desc0 + stage_off + (uint64_t)((k * 2048) >> 4),
                      b_desc0 + stage_off + (uint64_t)((k * 256) >> 4), idesc, (kb != kb0 || k != 0) ? 1u : 0u);
        tc_commit(&empty[stage]);
        stage_off += kStageStep;
        if (++stage == S) {
          stage = 0;
          stage_off = 0;
          phase ^= 1;
        }
      }
      if (ok) tc_commit(tfull);
      tc_commit(drain);
      mbar_wait(drain, 0, p.wait_ns, nullptr, nullptr);
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int k = mb * 128 + row;
    if (mbar_wait(tfull, 0, p.wait_ns, p.status, abort_flag)) {
      tc_fence_after();
      const long long dwsize = (long long)p.Cout * 72;
      const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
      float* o = p.part + (long long)split * dwsize + (long long)k * 72;
#pragma unroll 1
      for (int j = 0; j < 3; ++j) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(lane_addr + (uint32_t)(j * 32), v);
        tmem_ld_wait();
        if (k < p.Cout) {
          // column block qb (8 columns) holds tap qb; blocks 9-11 are the zero
          // and ones blocks
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int qb = 4 * j + g;
            if (qb < 9) {
              const int tap = qb;
              reinterpret_cast<float4*>(o + tap * 8)[0] =
                  make_float4(__uint_as_float(v[8 * g]), __uint_as_float(v[8 * g + 1]),
                              __uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]));
              reinterpret_cast<float4*>(o + tap * 8)[1] =
                  make_float4(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]),
                              __uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]));
            }
          }
          // column 80 (block 10) is the first ones column: dbias
          if (j == 2) p.part[(long long)p.S * dwsize + (long long)split * p.Cout + k] = __uint_as_float(v[16]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, 128);
}

// Width 64, x staged as three column-shifted copies of three halo rows.  x
// [N][H][64][8] is viewed as flat rows [N][H][512]; per 64-pixel k-block (one
// image row h) and column shift s = 0..2, two boxes of 256 elements x 3 rows
// (pixels 32 hf + s - 1 .. + 31 of rows h - 1 .. h + 1; outside the image
// reads zero) land at half hf's region + s * 1536, row r at + r * 512.  So in
// each half the 8-pixel x 16-byte core matrices of tap (r, s) start (3 s + r)
// * 512 bytes in: one uniform stride over the nine taps, and a static ones
// block at position 9 (dbias).  Per 16 pixels one M = 128, N = 80 MMA covers
// all nine taps where one copy per shift needed three N = 32 MMAs: measured on
// the 64x64 stem, the twelve small MMAs per k-block ran at the DRAM's pace and
// left no slack to drain the stages filled during the kernel's cold start.
constexpr uint32_t kWhHalf = 5120;                            // 9 row blocks + ones block, per half
constexpr uint32_t kWhX = kWgABytes;                          // x halves after dy
constexpr uint32_t kWhOnes = 9 * 512;                         // ones block within a half
constexpr uint32_t kWhStage = (kWhX + 2 * kWhHalf + 1023) / 1024 * 1024;
constexpr uint32_t kWhLoad = kWgABytes + 6 * 3 * 512;         // bytes copied per k-block
constexpr int kWhStages = 8;
constexpr size_t kWhSmem = (size_t)kWhStages * kWhStage + 256 + 1024;
static_assert(kWhStages >= kProd, "stage-parallel producers need S >= kProd");
static_assert(kWhX % 128 == 0 && kWhHalf % 16 == 0, "TMA destinations stay aligned");
static_assert(kWhSmem <= 227 * 1024, "shared memory per CTA");

__global__ void __launch_bounds__(kThreads, 1)
    k_wgrad_c8h(const __grid_constant__ CUtensorMap tmDY, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ CUtensorMap tmPart, const WgradParams p) {
  constexpr int S = kWhStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * kWhStage);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // no early trigger: the dependent is the partials' reduction
  const int mb = blockIdx.x % p.num_mb;
  const int split = blockIdx.x / p.num_mb;
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
  const int HW = p.H * p.W;

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmDY);
    tma_prefetch_desc(&tmX);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  if (warp >= kEpiBase) {  // every stage's two ones blocks (bf16 1.0 = 0x3F80)
    const int t = threadIdx.x - 32 * kEpiBase;
    for (int st = 0; st < S; ++st)
      for (int hf = 0; hf < 2; ++hf) {
        uint4* b = reinterpret_cast<uint4*>(smem + (size_t)st * kWhStage + kWhX + hf * kWhHalf + kWhOnes);
        for (int i = t; i < 512 / 16; i += 32 * kWgEpiWarps)
          b[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
      }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the previous kernel's writes are visible from here on

  if (warp < kProd) {
    // whole stages in turn: two dy boxes (64 pixels x 64 channels) and the
    // six x boxes of k-block kb (image row h0 of image n0)
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (issued % kProd == warp) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns, p.status, abort_flag)) {
            ok = false;
            break;
          }
          const int pk = kb * kWgPix;
          const int n0 = pk / HW, h0 = (pk - n0 * HW) / p.W;
          uint8_t* sa = smem + (size_t)stage * kWhStage;
          mbar_arrive_expect_tx(&full[stage], kWhLoad);
          tma_load_2d(sa, &tmDY, &full[stage], mb * 128, pk);
          tma_load_2d(sa + 8192, &tmDY, &full[stage], mb * 128 + 64, pk);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int sh = 0; sh < 3; ++sh)
              tma_load_3d(sa + kWhX + hf * kWhHalf + sh * 1536, &tmX, &full[stage], 256 * hf + 8 * (sh - 1),
                          h0 - 1, n0);
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        // wait (bounded) for the loads still in flight
        const int n = issued < S ? issued : S;
        for (int i = 0; i < n; ++i) {
          if (--stage < 0) {
            stage = S - 1;
            phase ^= 1;
          }
          mbar_wait(&full[stage], phase, drain_wait_ns(p.wait_ns), nullptr, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 80, 1, 1);
      // descriptors built once for stage 0; stages and K steps move the start
      // address only (addresses stay below 2^18: no carry)
      const uint32_t sbase = smem_u32(smem);
      const uint64_t a_desc0 = smem_desc(sbase, 8192, 1024, kSwizzle128B);
      const uint64_t x_desc0 = smem_desc(sbase + kWhX, 128, 512, kSwizzleNone);
      constexpr uint32_t kStageStep = kWhStage >> 4;
      int stage = 0;
      uint32_t phase = 0, stage_off = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full[stage], phase, p.wait_ns, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad0 = a_desc0 + stage_off, xd0 = x_desc0 + stage_off;
#pragma unroll
        for (int k = 0; k < kWgPix / 16; ++k)
          tc_mma_bf16(tmem_base, ad0 + (uint64_t)((k * 2048) >> 4),
                      xd0 + (uint64_t)(((k >> 1) * kWhHalf + (k & 1) * 256) >> 4), idesc,
                      (kb != kb0 || k != 0) ? 1u : 0u);
        tc_commit(&empty[stage]);
        stage_off += kStageStep;
        if (++stage == S) {
          stage = 0;
          stage_off = 0;
          phase ^= 1;
        }
      }
      if (ok) tc_commit(tfull);
      tc_commit(drain);
      mbar_wait(drain, 0, p.wait_ns, nullptr, nullptr);
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int k = mb * 128 + row;
    if (mbar_wait(tfull, 0, p.wait_ns, p.status, abort_flag)) {
      tc_fence_after();
      const long long dwsize = (long long)p.Cout * 72;
      const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
      // the partial row of channel k: in global memory, or (part_tma) row
      // `lane` of this warp's 32 x 72-float box in the idle stage memory,
      // stored with one TMA tensor store (rows past Cout are clipped)
      float* o = p.part_tma ? reinterpret_cast<float*>(smem + (size_t)q * 32 * 288) + lane * 72
                            : p.part + (long long)split * dwsize + (long long)k * 72;
#pragma unroll 1
      for (int c = 0; c < 3; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(lane_addr + (uint32_t)(32 * c), v);
        tmem_ld_wait();
        if (p.part_tma || k < p.Cout) {
          // column block j = 3 s + r (8 columns) holds tap (r, s)
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int j = 4 * c + g;
            if (j < 9) {
              const int tap = 3 * (j % 3) + j / 3;
              reinterpret_cast<float4*>(o + tap * 8)[0] =
                  make_float4(__uint_as_float(v[8 * g]), __uint_as_float(v[8 * g + 1]),
                              __uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]));
              reinterpret_cast<float4*>(o + tap * 8)[1] =
                  make_float4(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]),
                              __uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]));
            }
          }
          // column 72 (block 9, the ones block) is dbias
          if (c == 2 && k < p.Cout)
            p.part[(long long)p.S * dwsize + (long long)split * p.Cout + k] = __uint_as_float(v[8]);
        }
      }
      if (p.part_tma) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (mb * 128 + q * 32 < p.Cout)
            tma_store_3d(&tmPart, smem + (size_t)q * 32 * 288, 0, mb * 128 + q * 32, split);
          bulk_commit();
          bulk_wait_read<0>();  // the store's writes complete with the grid
        }
        __syncwarp();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, 128);
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
// NHWC activations as an im2col map.  Default: window origins run over
// [-1, size - 2] (pad 1, 3 taps) in steps of `ustride` (1, or 2 for a
// stride-2 conv: origins -1, 1, 3, ...).  corner = 0: origins over
// [0, size - 1] with offsets 0..1 (the 2x2 windows of the stride-2 dgrad).
int make_im2col_map(CUtensorMap* m, const void* base, int N, int H, int W, int C, int pixels,
                    int channels = BKC, bool swizzle = true, int ustride = 1, int corner = -1) {
  PFN_encodeIm2col enc = encode_im2col_fn();
  if (!enc) return CONV3X3_ERR_CUDA;
  cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)N};
  cuuint64_t strides[3] = {(cuuint64_t)C * 2, (cuuint64_t)W * C * 2, (cuuint64_t)H * W * C * 2};
  int lower[2] = {corner, corner};
  int upper[2] = {corner, corner};
  cuuint32_t estr[4] = {1, (cuuint32_t)ustride, (cuuint32_t)ustride, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                   lower, upper, (cuuint32_t)channels, (cuuint32_t)pixels, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

// NHWC activations as a tiled 4-D map; box {64 channels, box_w (default W)
// columns, rows, 1 image}.
// Boxes may start at w = -1 or h = -1 and run past the far edge: those
// elements read as zero (the convolution's padding).
int make_halo_map(CUtensorMap* m, const void* base, int N, int H, int W, int C, int rows,
                  int box_w = 0) {
  PFN_encodeTiled enc = encode_tiled_fn();
  if (!enc) return CONV3X3_ERR_CUDA;
  cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)N};
  cuuint64_t strides[3] = {(cuuint64_t)C * 2, (cuuint64_t)W * C * 2, (cuuint64_t)H * W * C * 2};
  cuuint32_t box[4] = {(cuuint32_t)BKC, (cuuint32_t)(box_w ? box_w : W), (cuuint32_t)rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

// KRSC weights viewed as {Cin, 9, Cout}; box {64, 1, rows}.
int make_weight_map(CUtensorMap* m, const void* w, int Cin, int Cout, int rows, int channels = BKC,
                    bool swizzle = true) {
  PFN_encodeTiled enc = encode_tiled_fn();
  if (!enc) return CONV3X3_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)Cin, 9, (cuuint64_t)Cout};
  cuuint64_t strides[2] = {(cuuint64_t)Cin * 2, (cuuint64_t)Cin * 9 * 2};
  cuuint32_t box[3] = {(cuuint32_t)channels, 1, (cuuint32_t)rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

// [P][C] activations as a 2-D map, box {64 channels, 64 pixels}.
int make_rows_map(CUtensorMap* m, const void* base, long long P, int C) {
  PFN_encodeTiled enc = encode_tiled_fn();
  if (!enc) return CONV3X3_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)P};
  cuuint64_t strides[1] = {(cuuint64_t)C * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kWgPix};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

template <typename K>
int set_smem(K kernel, size_t bytes, int device) {
  // cudaFuncSetAttribute once per (kernel, device); devices up to 64.
  static std::mutex mu;
  static uint64_t done[64] = {0};
  static const void* keys[64] = {nullptr};
  std::lock_guard<std::mutex> g(mu);
  int slot = -1;
  for (int i = 0; i < 64; ++i) {
    if (keys[i] == (const void*)kernel) {
      slot = i;
      break;
    }
    if (keys[i] == nullptr) {
      keys[i] = (const void*)kernel;
      slot = i;
      break;
    }
  }
  if (slot >= 0 && device >= 0 && device < 64 && (done[slot] >> device & 1)) return CONV3X3_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
      cudaSuccess)
    return CONV3X3_ERR_CUDA;
  if (slot >= 0 && device >= 0 && device < 64) done[slot] |= 1ull << device;
  return CONV3X3_OK;
}

// The TMA-store epilogue (IgemmParams::epi_tma) for a plain bf16 output:
// every tile where every CTA or pair has one (1), else each CTA's or pair's
// last tile (2), whose epilogue otherwise runs exposed at the end of the
// launch; `ty` then maps the output.  CONV3X3_EPI_TMA=0 keeps the per-thread
// row stores everywhere, CONV3X3_EPI_TMA=1 uses TMA stores on one-tile
// launches only.
int make_store_map(CUtensorMap* m, void* base, long long P, int C);
void epi_tma_setup(IgemmParams& p, bool allowed, int tiles, int slots, const CUtensorMap& dummy,
                   CUtensorMap* ty) {
  *ty = dummy;
  p.epi_tma = 0;
  if (!allowed || p.out_f32 || p.zout || p.out2 || p.s2 || p.nsplit != p.nout || p.nout % 8) return;
  const int mode = tiles > slots ? 2 : 1;
  if (const char* e = std::getenv("CONV3X3_EPI_TMA")) {
    if (std::strcmp(e, "0") == 0) return;
    if (std::strcmp(e, "1") == 0 && mode == 2) return;
  }
  if (make_store_map(ty, p.out, p.P, p.nout) == CONV3X3_OK) p.epi_tma = mode;
}

template <int BN, int MT, bool kDgrad, int KC = 1, bool kT = false>
int launch_igemm(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b,
                 const IgemmParams& prm, const DevCtx& d, cudaStream_t st) {
  using Cfg = IgemmCfg<BN, MT, KC>;
  // the fused extras, a split output or a stride-2 dgrad need the full epilogue
  const bool ext = prm.zout || prm.zin || prm.out2 || prm.s2;
  auto kern = ext ? k_igemm<BN, MT, kDgrad, true, KC, kT> : k_igemm<BN, MT, kDgrad, false, KC, kT>;
  if (set_smem(kern, Cfg::kSmem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
  const int tiles = (prm.s2 ? 4 : 1) * prm.num_m_tiles * prm.num_n_tiles;
  const int grid = tiles < d.num_sms ? tiles : d.num_sms;
  IgemmParams p2 = prm;
  CUtensorMap ty;
  epi_tma_setup(p2, !kT, tiles, grid, a, &ty);  // (the transposed tile has its own epilogue)
  launch_pdl(kern, dim3(grid), dim3(igemm_threads(kT && ext)), Cfg::kSmem, st, a, a2, b, ty, p2);
  return cudaGetLastError() == cudaSuccess ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

// Resident clusters of `csize` CTAs (two for k_igemm_pair, four for
// k_igemm_pks; a GPC whose free SMs are not a multiple of the cluster size
// leaves some idle), cached per kernel and device.
template <typename K>
int pair_slots(K kernel, size_t smem, const DevCtx& d, int csize = 2) {
  constexpr int kKeys = 16;
  static std::mutex mu;
  static int cache[kKeys][64] = {};
  static const void* keys[kKeys] = {};
  std::lock_guard<std::mutex> g(mu);
  int slot = 0;
  while (slot < kKeys && keys[slot] != nullptr && keys[slot] != (const void*)kernel) ++slot;
  const bool cacheable = slot < kKeys && d.device >= 0 && d.device < 64;
  if (cacheable && keys[slot] == (const void*)kernel && cache[slot][d.device] > 0)
    return cache[slot][d.device];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize * (d.num_sms / csize), 1, 1);
  cfg.blockDim = dim3(kIgemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    n = d.num_sms / csize;
  }
  if (cacheable) {
    keys[slot] = (const void*)kernel;
    cache[slot][d.device] = n;
  }
  return n;
}

// First work item of the half-width tiles of a 256-channel pair launch (see
// IgemmParams::half_from), or INT_MAX for none.  Where the tiles leave a last
// round that fills at most half of the pairs, that round's tiles run as two
// 128-channel items each: they then spread over up to all of the pairs and
// the round takes a half-width item's time.  CONV3X3_PAIR_HALF=0 keeps whole
// tiles; CONV3X3_PAIR_HALF=all splits every tile (tests).
int pair_half_from(int tiles, int pairs) {
  int mode = -1;
  if (const char* e = std::getenv("CONV3X3_PAIR_HALF")) mode = std::strcmp(e, "all") == 0 ? 1 : 0;
  if (mode == 1) return 0;
  if (mode == 0 || tiles <= pairs) return 0x7fffffff;
  const int whole = tiles / pairs * pairs, left = tiles - whole;
  return left > 0 && 2 * left <= pairs ? whole : 0x7fffffff;
}

template <bool kDgrad, int BN, int KC = 1>
int launch_igemm_pair(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b,
                      const CUtensorMap& b64, const IgemmParams& prm, const DevCtx& d,
                      cudaStream_t st) {
  using Cfg = PairCfg<BN, kDgrad, KC>;
  const bool ext = prm.zout || prm.zin || prm.out2;
  auto kern = ext ? k_igemm_pair<kDgrad, true, BN, KC> : k_igemm_pair<kDgrad, false, BN, KC>;
  if (set_smem(kern, Cfg::kSmem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
  const int tiles = prm.num_m_tiles * prm.num_n_tiles;
  const int pairs = pair_slots(kern, Cfg::kSmem, d);
  IgemmParams p2 = prm;
  p2.half_from = BN == 256 ? pair_half_from(tiles, pairs) : 0x7fffffff;
  const int items = p2.half_from < tiles ? 2 * tiles - p2.half_from : tiles;
  const int grid = 2 * (items < pairs ? items : pairs);
  CUtensorMap ty;
  epi_tma_setup(p2, true, items, grid / 2, a, &ty);
  launch_pdl(kern, dim3(grid), dim3(kIgemmThreads), Cfg::kSmem, st, a, a2, b, b64, ty, p2);
  return cudaGetLastError() == cudaSuccess ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

template <bool kDgrad>
int launch_igemm_ks(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b,
                    const IgemmParams& prm, const DevCtx& d, cudaStream_t st) {
  const bool ext = prm.zout || prm.zin || prm.out2;
  auto kern = ext ? k_igemm_ks<kDgrad, true> : k_igemm_ks<kDgrad, false>;
  if (set_smem(kern, kKsSmem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
  const int grid = 2 * prm.num_m_tiles * prm.num_n_tiles;  // one tile per cluster
  launch_pdl(kern, dim3(grid), dim3(kIgemmThreads), kKsSmem, st, a, a2, b, prm);
  return cudaGetLastError() == cudaSuccess ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

// K split over two pairs: one 256 x 256 tile per cluster of four.  Returns
// CONV3X3_ERR_UNSUPPORTED (nothing launched) where the tiles' clusters do not
// all fit on the GPU at once.
template <bool kDgrad>
int launch_igemm_pks(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b,
                     const IgemmParams& prm, const DevCtx& d, cudaStream_t st) {
  using Cfg = PairCfg<kPksBN, kDgrad, kPksKC>;
  const bool ext = prm.zout || prm.zin || prm.out2;
  auto kern = ext ? k_igemm_pks<kDgrad, true> : k_igemm_pks<kDgrad, false>;
  if (set_smem(kern, Cfg::kSmem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
  const int tiles = prm.num_m_tiles * prm.num_n_tiles;
  if (tiles > pair_slots(kern, Cfg::kSmem, d, 4)) return CONV3X3_ERR_UNSUPPORTED;
  launch_pdl(kern, dim3(4 * tiles), dim3(kIgemmThreads), Cfg::kSmem, st, a, a2, b, prm);
  return cudaGetLastError() == cudaSuccess ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

template <int W_, int BN, bool kDgrad>
int launch_halo(const CUtensorMap& a, const CUtensorMap& b, const IgemmParams& prm,
                const DevCtx& d, cudaStream_t st) {
  using Cfg = HaloCfg<W_, BN>;
  auto kern = k_halo<W_, BN, kDgrad>;
  if (set_smem(kern, Cfg::kSmem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
  const int tiles = prm.num_m_tiles * prm.num_n_tiles;
  const int grid = tiles < d.num_sms ? tiles : d.num_sms;
  launch_pdl(kern, dim3(grid), dim3(kIgemmThreads), Cfg::kSmem, st, a, b, prm);
  return cudaGetLastError() == cudaSuccess ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

struct TileShape {
  int bn, mt;
  bool halo;
};

// Tile choice.  Per 64-channel k-block a CTA tile of (128*MT) pixels x BN
// channels stages (128*MT + BN) * 128 bytes into shared memory and keeps the
// tensor core busy MT * BN / 128 * 256 cycles.  The stage ring (~200 KB) turns
// over once per MMA-completion + TMA round trip (~2500 cycles), which caps
// delivery near 80 B per cycle per SM; the k-block time is the larger of the
// two.  Score = persistent-tile rounds x k-block time; near-ties go to the
// tile listed first (larger).
TileShape pick_tile(int nout, const Shape& sh, int num_sms) {
  const long long P = sh.P();
  const TileShape cand[6] = {{256, 1, false}, {128, 2, false}, {192, 1, false},
                             {128, 1, false}, {64, 2, false}, {64, 1, false}};
  TileShape best = {128, 1, false};
  double best_cost = -1.0;
  // Halo tiles (256 pixels = whole rows of one image, BN <= 128) stage a
  // third of the im2col bytes, but measured slower than the im2col kernels on
  // GB300 (the copies, not the bytes, set the pace); they stay selectable
  // through CONV3X3_TILE and are not scored here.
  if (false && (sh.W == 16 || sh.W == 32 || sh.W == 64) && sh.H % (256 / sh.W) == 0) {
    const int bn = nout > 64 ? 128 : 64;
    const long long n_tiles = (nout + bn - 1) / bn;
    const long long waste = n_tiles * bn - nout;
    if (bn == 64 || waste * 2 <= bn) {
      const long long rounds = (P / 256 * n_tiles + num_sms - 1) / num_sms;
      const double mma = 512.0 * bn / 128.0;
      const double a_bytes = 3.0 * (256 + 2 * sh.W) * 128.0;
      const double feed = (a_bytes + 9.0 * bn * 128.0) / 9.0 / 80.0;
      best_cost = (double)rounds * (mma > feed ? mma : feed);
      best = {bn, 2, true};
    }
  }
  for (int i = 0; i < 6; ++i) {
    const TileShape c = cand[i];
    const long long n_tiles = (nout + c.bn - 1) / c.bn;
    const long long waste = n_tiles * c.bn - nout;
    if (c.bn > 64 && waste * 2 > c.bn) continue;  // mostly-empty last tile
    const long long m_tiles = (P + 128LL * c.mt - 1) / (128LL * c.mt);
    const long long rounds = (m_tiles * n_tiles + num_sms - 1) / num_sms;
    const double mma = 256.0 * c.mt * c.bn / 128.0;
    const double feed = (128.0 * c.mt + c.bn) * 128.0 / 80.0;
    const double cost = (double)rounds * (mma > feed ? mma : feed);
    if (best_cost < 0 || cost < 0.97 * best_cost) {
      best_cost = cost;
      best = c;
    }
  }
  return best;
}

template <int BN, bool kTS = false, int kRW = 0, bool kZ = false>
int launch_stem(const CUtensorMap& a, const __nv_bfloat16* w, const CUtensorMap& y, const CUtensorMap& z,
                const IgemmParams& prm, const DevCtx& d, cudaStream_t st) {
  using Cfg = StemCfg<BN, kTS, kRW, kZ>;
  auto kern = k_stem_fwd<BN, kTS, kRW, kZ>;
  if (set_smem(kern, Cfg::kSmem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
  const int grid = prm.num_m_tiles < d.num_sms ? prm.num_m_tiles : d.num_sms;
  launch_pdl(kern, dim3(grid), dim3(kIgemmThreads), Cfg::kSmem, st, a, w, y, z, prm);
  return cudaGetLastError() == cudaSuccess ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

// [P][C] bf16 output as a 2-D map for TMA stores: box {64 channels, 32 pixels},
// 128-byte swizzle (the staging layout of the TMA-store epilogues).
int make_store_map(CUtensorMap* m, void* base, long long P, int C) {
  PFN_encodeTiled enc = encode_tiled_fn();
  if (!enc) return CONV3X3_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)P};
  cuuint64_t strides[1] = {(cuuint64_t)C * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

// x [N][H][W][8] viewed as [N][H][W * 8]: boxes of `elems` consecutive
// elements of `rows` image rows (no swizzle), for the row-staged 8-channel
// kernels.
int make_row_map(CUtensorMap* m, const void* base, int N, int H, int W, int elems, int rows = 1) {
  PFN_encodeTiled enc = encode_tiled_fn();
  if (!enc) return CONV3X3_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)W * 8, (cuuint64_t)H, (cuuint64_t)N};
  cuuint64_t strides[2] = {(cuuint64_t)W * 16, (cuuint64_t)H * W * 16};
  cuuint32_t box[3] = {(cuuint32_t)elems, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

// Row staging for the 8-channel forward: width 32 or 64 and 128-pixel tiles of
// whole image rows of one image.  CONV3X3_STEM_ROWS=0 keeps im2col boxes.
int stem_row_width(const Shape& s) {
  if (const char* e = std::getenv("CONV3X3_STEM_ROWS"))
    if (std::strcmp(e, "0") == 0) return 0;
  if (s.u != 1 || !(s.W == 32 || s.W == 64)) return 0;
  return ((long long)s.H * s.W) % BM == 0 ? s.W : 0;
}

// Forward with exactly 8 input channels and at most 256 outputs (one N tile).
int run_stem_fwd(const void* x, const void* w, const float* bias, void* y, const Shape& s, int act,
                 int out_f32, const EpiExtra& ex, const DevCtx& d, cudaStream_t st) {
  const int bn = s.Cout <= 64 ? 64 : s.Cout <= 128 ? 128 : 256;
  const int rw = stem_row_width(s);
  CUtensorMap ta;
  int rc = rw ? make_row_map(&ta, x, s.N, s.H, s.W, rw * 8 < 256 ? rw * 8 : 256)
              : make_im2col_map(&ta, x, s.N, s.H, s.W, 8, BM, 8, false);
  if (rc) return rc;
  const __nv_bfloat16* wp = static_cast<const __nv_bfloat16*>(w);
  IgemmParams prm;
  prm.out = y;
  prm.bias = bias;
  prm.act = act;
  prm.out_f32 = out_f32;
  prm.P = (int)s.P();
  prm.H = s.H;
  prm.W = s.W;
  prm.kchunks = 1;
  prm.kgroups = 1;
  prm.kchunks_a = 1;
  prm.ustride = 1;
  prm.s2 = 0;
  prm.oh = s.H;
  prm.ow = s.W;
  prm.nout = s.Cout;
  prm.nsplit = s.Cout;
  prm.num_m_tiles = (int)((s.P() + BM - 1) / BM);
  prm.num_n_tiles = 1;
  prm.status = d.status;
  prm.wait_ns = d.wait_ns;
  prm.zout = static_cast<__nv_bfloat16*>(ex.zout);
#define C3_STEM(BN_, TS_, Y_)                                                  \
  return rw == 64   ? launch_stem<BN_, TS_, 64>(ta, wp, Y_, ta, prm, d, st)      \
         : rw == 32 ? launch_stem<BN_, TS_, 32>(ta, wp, Y_, ta, prm, d, st)      \
                    : launch_stem<BN_, TS_, 0>(ta, wp, Y_, ta, prm, d, st)
  if (bn == 128 && !out_f32 && !ex.zout) {
    // bf16 output with no z store leaves through TMA stores
    CUtensorMap ty;
    rc = make_store_map(&ty, y, s.P(), s.Cout);
    if (rc) return rc;
    C3_STEM(128, true, ty);
  }
  if (bn == 128 && !out_f32 && ex.zout && rw) {
    // and with the z store (row staging): both through TMA stores.
    // CONV3X3_STEM_ZTMA=0 keeps per-thread stores for both.
    const char* e = std::getenv("CONV3X3_STEM_ZTMA");
    if (!(e && std::strcmp(e, "0") == 0)) {
      CUtensorMap ty, tz;
      rc = make_store_map(&ty, y, s.P(), s.Cout);
      if (rc) return rc;
      rc = make_store_map(&tz, ex.zout, s.P(), s.Cout);
      if (rc) return rc;
      return rw == 64 ? launch_stem<128, true, 64, true>(ta, wp, ty, tz, prm, d, st)
                      : launch_stem<128, true, 32, true>(ta, wp, ty, tz, prm, d, st);
    }
  }
  // (without TMA stores the output map is unused: ta stands in)
  if (bn == 64) C3_STEM(64, false, ta);
  if (bn == 128) C3_STEM(128, false, ta);
  C3_STEM(256, false, ta);
#undef C3_STEM
}

// dgrad with 8 output channels (k_stem_dgrad): whole-row tiles of 128 dx
// pixels, dy channels a multiple of 64 up to 128.
bool stem_dgrad_fits(const Shape& s) {
  if (s.Cin != 8 || s.u != 1 || s.Cout % 64 != 0 || s.Cout > 128) return false;
  if (s.W > 64 || BM % s.W != 0) return false;
  const int R = BM / s.W;
  return R <= s.H && s.H % R == 0;
}

// Width 64, row bands (k_stem_dgrad_rows): selected by CONV3X3_STEM_DGRAD=rows.
// Measured on GB300 (batch 64, 64x64, 128 dy channels) it ran in 32.8 us
// against 28.7 us for the tile kernel: both are bound by the epilogue's
// per-chunk round trip (stage T, synchronise, sum, synchronise), and a band
// walked in order gives each round trip one or two dx rows where a tile gives
// two, so the halved tensor and copy work did not pay.
int run_stem_dgrad_rows(const void* dy, const void* w, void* dx, const Shape& s, int out_f32,
                        const EpiExtra& ex, const DevCtx& d, cudaStream_t st) {
  PFN_encodeTiled enc = encode_tiled_fn();
  if (!enc) return CONV3X3_ERR_CUDA;
  // dy as [N * H][64][K]: boxes of 64 channels x 64 pixels x 2 rows
  CUtensorMap tdy;
  const int NH = s.N * s.H;
  cuuint64_t dims[3] = {(cuuint64_t)s.Cout, (cuuint64_t)kSrW, (cuuint64_t)NH};
  cuuint64_t strides[2] = {(cuuint64_t)s.Cout * 2, (cuuint64_t)kSrW * s.Cout * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kSrW, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&tdy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(dy), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return CONV3X3_ERR_CUDA;
  StemDgradRowsParams prm;
  prm.out = dx;
  prm.out_f32 = out_f32;
  prm.zin = static_cast<const __nv_bfloat16*>(ex.zin);
  prm.zin_act = ex.zin ? ex.zin_act : CONV3X3_ACT_NONE;
  prm.NH = NH;
  prm.H = s.H;
  prm.K = s.Cout;
  const int grid0 = NH < d.num_sms ? NH : d.num_sms;
  prm.band = (NH + grid0 - 1) / grid0;
  const int grid = (NH + prm.band - 1) / prm.band;
  prm.status = d.status;
  prm.wait_ns = d.wait_ns;
  const size_t smem = stem_dgrad_rows_smem(s.Cout);
  if (set_smem(k_stem_dgrad_rows, smem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
  launch_pdl(k_stem_dgrad_rows, dim3(grid), dim3(kSdThreads), smem, st, tdy,
             static_cast<const __nv_bfloat16*>(w), prm);
  return cudaGetLastError() == cudaSuccess ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

int run_stem_dgrad(const void* dy, const void* w, void* dx, const Shape& s, int out_f32,
                   const EpiExtra& ex, const DevCtx& d, cudaStream_t st) {
  const char* e = std::getenv("CONV3X3_STEM_DGRAD");
  if (s.W == kSrW && e && std::strcmp(e, "rows") == 0)
    return run_stem_dgrad_rows(dy, w, dx, s, out_f32, ex, d, st);
  PFN_encodeTiled enc = encode_tiled_fn();
  if (!enc) return CONV3X3_ERR_CUDA;
  const int R = BM / s.W;
  CUtensorMap tdy;
  cuuint64_t dims[4] = {(cuuint64_t)s.Cout, (cuuint64_t)s.W, (cuuint64_t)s.H, (cuuint64_t)s.N};
  cuuint64_t strides[3] = {(cuuint64_t)s.Cout * 2, (cuuint64_t)s.W * s.Cout * 2,
                           (cuuint64_t)s.H * s.W * s.Cout * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)s.W, (cuuint32_t)(R + 2), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (enc(&tdy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(dy), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return CONV3X3_ERR_CUDA;
  StemDgradParams prm;
  prm.out = dx;
  prm.out_f32 = out_f32;
  prm.zin = static_cast<const __nv_bfloat16*>(ex.zin);
  prm.zin_act = ex.zin ? ex.zin_act : CONV3X3_ACT_NONE;
  prm.P = (int)s.P();
  prm.H = s.H;
  prm.W = s.W;
  prm.K = s.Cout;
  prm.R = R;
  prm.num_tiles = s.N * (s.H / R);
  prm.status = d.status;
  prm.wait_ns = d.wait_ns;
  const size_t smem = stem_dgrad_smem(s.Cout);
  if (set_smem(k_stem_dgrad, smem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
  const int grid = prm.num_tiles < d.num_sms ? prm.num_tiles : d.num_sms;
  launch_pdl(k_stem_dgrad, dim3(grid), dim3(kSdThreads), smem, st, tdy,
             static_cast<const __nv_bfloat16*>(w), prm);
  return cudaGetLastError() == cudaSuccess ? CONV3X3_OK : CONV3X3_ERR_CUDA;
}

// Forward (a_src = x, a_ch = Cin) or dgrad (a_src = dy, a_ch = Cout).  With a
// channel split the forward reads x's channels [Ca, Cin) from cat.b and the
// dgrad writes dx's channels [Ca, Cin) to cat.b.
int run_igemm(bool dgrad, const void* a_src, int a_ch, const void* w, const float* bias, void* out,
              const Shape& s, int act, int out_f32, const EpiExtra& ex, const CatSplit& cat,
              const DevCtx& d, cudaStream_t st) {
  const int nout = dgrad ? s.Cin : s.Cout;
  // pixel grid the tiles traverse: y's (forward), dx's (stride-1 dgrad) or
  // dy's (stride-2 dgrad, four parity classes over it)
  const bool s2 = dgrad && s.u == 2;
  Shape g = s;
  if (!dgrad || s2) {
    g.H = s.Ho();
    g.W = s.Wo();
  }
  g.u = 1;
  TileShape ts = pick_tile(nout, dgrad ? s : g, d.num_sms);
  // 128-channel x 256-pixel tiles run transposed (k_igemm kT) unless the
  // override names "128x2n".  256-channel tiles run on CTA pairs
  // (k_igemm_pair) where that measured faster: a forward of at least two
  // 64-channel chunks with at least two rounds of pair tiles (a 256-pixel pair
  // tile halves the tile count, so small grids lose; 128 -> 256 channels at
  // 32x32: 39.8 -> 37.5 us), or a dgrad whose pair tiles fill at least 4/5 of
  // the SMs (1024 -> 512 at 8x8 and 256 -> 384 at 16x16, 64 pair tiles each:
  // 33.7 -> 33.0 and 29.3 -> 27.5 us; 32 pair tiles ran slower).
  // CONV3X3_PAIR=0|1 or the override "256x1" / "256x1n" forces the choice.
  bool trans = true;
  int pair_force = -1, pair_bn = 0;
  if (const char* e = std::getenv("CONV3X3_PAIR")) pair_force = std::strcmp(e, "0") != 0 ? 1 : 0;
  // CONV3X3_TILE="<BN>x<MT>", "halo<BN>" or "pair<BN>" overrides the choice (tuning and tests)
  if (const char* e = std::getenv("CONV3X3_TILE")) {
    trans = std::strcmp(e, "128x2n") != 0;
    if (std::strcmp(e, "256x1n") == 0) pair_force = 0;
    if (std::strcmp(e, "256x1") == 0) pair_force = 1;
    int pb = 0;
    if (std::sscanf(e, "pair%d", &pb) == 1 && (pb == 128 || pb == 192 || pb == 256 || pb == 384)) pair_bn = pb;
    int bn_o = 0, mt_o = 0;
    const bool halo_ok = (s.W == 16 || s.W == 32 || s.W == 64) && s.H % (256 / s.W) == 0;
    if (std::sscanf(e, "halo%d", &bn_o) == 1 && halo_ok && (bn_o == 64 || bn_o == 128))
      ts = TileShape{bn_o, 2, true};
    else if (std::sscanf(e, "%dx%d", &bn_o, &mt_o) == 2 && (mt_o == 1 || mt_o == 2) &&
             (bn_o == 64 || bn_o == 128 || bn_o == 192 || bn_o == 256) && 2 * mt_o * bn_o <= 512)
      ts = TileShape{bn_o, mt_o, false};
  }
  if (ts.halo && (cat.on() || s.u != 1))  // the halo kernel reads one stride-1 tensor
    ts = pick_tile(nout, dgrad ? s : g, d.num_sms);
  const int bn = ts.bn;
  const bool split_a = cat.on() && !dgrad;  // forward: A comes from two tensors
  const int a_ch1 = split_a ? cat.Ca : a_ch;
  CUtensorMap ta, ta2, tb;
  // A: x over its own grid with the conv's stride (forward), dy over dx's grid
  // (stride-1 dgrad) or over its own grid in 2x2 windows (stride-2 dgrad)
  const int a_h = dgrad ? g.H : s.H, a_w = dgrad ? g.W : s.W;
  const int a_u = dgrad ? 1 : s.u, a_corner = s2 ? 0 : -1;
  int rc = ts.halo ? make_halo_map(&ta, a_src, s.N, s.H, s.W, a_ch, (256 / s.W + 2) / 2)
                   : make_im2col_map(&ta, a_src, s.N, a_h, a_w, a_ch1, BM, BKC, true, a_u, a_corner);
  if (rc) return rc;
  if (split_a) {
    rc = make_im2col_map(&ta2, cat.b, s.N, s.H, s.W, a_ch - cat.Ca, BM, BKC, true, a_u, a_corner);
    if (rc) return rc;
  } else {
    ta2 = ta;
  }
  rc = make_weight_map(&tb, w, s.Cin, s.Cout, (kOneWeightBox && !dgrad && !ts.halo) ? bn : 64);
  if (rc) return rc;
  IgemmParams prm;
  prm.out = out;
  prm.bias = bias;
  prm.act = act;
  prm.out_f32 = out_f32;
  prm.P = (int)g.P();
  prm.H = g.H;
  prm.W = g.W;
  prm.ustride = dgrad ? 1 : s.u;
  prm.s2 = s2 ? 1 : 0;
  prm.oh = s.H;
  prm.ow = s.W;
  prm.kchunks_a = split_a ? cat.Ca / BKC : (a_ch + BKC - 1) / BKC;
  prm.kchunks = split_a ? prm.kchunks_a + (a_ch - cat.Ca + BKC - 1) / BKC : prm.kchunks_a;
  prm.kgroups = prm.kchunks;
  prm.nout = nout;
  prm.nsplit = (cat.on() && dgrad) ? cat.Ca : nout;
  prm.out2 = (cat.on() && dgrad) ? cat.b : nullptr;
  prm.num_m_tiles = (int)((g.P() + BM * ts.mt - 1) / (BM * ts.mt));
  prm.num_n_tiles = (nout + bn - 1) / bn;
  prm.status = d.status;
  prm.wait_ns = d.wait_ns;
  prm.zout = static_cast<__nv_bfloat16*>(ex.zout);
  prm.zin = static_cast<const __nv_bfloat16*>(ex.zin);
  prm.zin2 = static_cast<const __nv_bfloat16*>(ex.zin_b);
  prm.zin_act = ex.zin ? ex.zin_act : CONV3X3_ACT_NONE;
  if (ts.halo) {
#define C3_HALO(W_, BN_) \
  return dgrad ? launch_halo<W_, BN_, true>(ta, tb, prm, d, st) : launch_halo<W_, BN_, false>(ta, tb, prm, d, st)
    if (s.W == 64) {
      if (bn == 64) C3_HALO(64, 64);
      C3_HALO(64, 128);
    }
    if (s.W == 32) {
      if (bn == 64) C3_HALO(32, 64);
      C3_HALO(32, 128);
    }
    if (bn == 64) C3_HALO(16, 64);
    C3_HALO(16, 128);
#undef C3_HALO
  }
  const long long pair_tiles = (g.P() + 2 * BM - 1) / (2 * BM) * prm.num_n_tiles;
  const bool pair = pair_force >= 0 ? pair_force == 1
                    : dgrad ? 10 * pair_tiles >= 4LL * d.num_sms
                            : (prm.kchunks >= 2 && pair_tiles >= d.num_sms);
  if (pair_bn == 0 && pair && bn == 256 && ts.mt == 1) pair_bn = 256;
  // 384 output channels whose 256-pixel x 384-channel pair tiles fill most of
  // the GPU in one round, with a K of at least four 64-channel chunks: one tile
  // per cluster, an N = 256 and an N = 128 MMA per K step.  Measured on GB300 (batch 64,
  // 16x16): 896 -> 384 forward 79.6 -> 71.5 us, 384 -> 384 dgrad 40.8 -> 38.9
  // us against 128 x 192 one-CTA tiles; 256 -> 384 (four chunks) 33.0 -> 29.9
  // us once the one-tile epilogue stored through TMA; 16 pair tiles (8x8) ran
  // slower.  CONV3X3_PAIR384=0 keeps the tile choice above.
  const long long tiles384 = (g.P() + 2 * BM - 1) / (2 * BM);
  bool p384 = pair_bn == 0 && pair_force != 0 && nout == 384 && tiles384 <= d.num_sms / 2 &&
              tiles384 * 8 >= 3LL * d.num_sms && prm.kchunks >= 4;
  if (const char* e = std::getenv("CONV3X3_PAIR384"))
    if (std::strcmp(e, "0") == 0) p384 = false;
  if (p384) pair_bn = 384;
  // K split over two pairs (k_igemm_pks) where 256 x 256 pair tiles would
  // leave most pairs idle but their clusters of four fill at least half of
  // the GPU at once, with an even input chunk count (two chunks per stage) of
  // at least eight: the 8x8 layers of 512 output channels.  Measured on GB300
  // (batch 64, 8x8, per call): 1024 -> 512 forward 39.4 -> 35.1 us against
  // the one-CTA K split, 512 -> 512 dgrad 25.0 -> 24.5 us and forward equal
  // against 128 x 128 tiles; 384 -> 512 (six chunks) 20.8 -> 22.8 us, so it
  // keeps 128 x 128 tiles.  Not under a forced tile (CONV3X3_TILE);
  // CONV3X3_PKS=0|1 forbids it, or takes it wherever the shape allows (at
  // least four chunks) and the clusters fit.
  const long long pks_tiles = (g.P() + 2 * BM - 1) / (2 * BM) * ((nout + kPksBN - 1) / kPksBN);
  const bool pks_shape = !s2 && !ts.halo && pair_bn == 0 && nout % kPksBN == 0 && prm.kchunks % 2 == 0 &&
                         prm.kchunks >= 4;
  bool pks = pks_shape && prm.kchunks >= 8 && std::getenv("CONV3X3_TILE") == nullptr &&
             4 * pks_tiles <= d.num_sms && 8 * pks_tiles >= d.num_sms;
  if (const char* e = std::getenv("CONV3X3_PKS")) pks = std::strcmp(e, "0") != 0 && pks_shape;
  if (pks) {
    IgemmParams pq = prm;
    pq.num_m_tiles = (int)((g.P() + 2 * BM - 1) / (2 * BM));
    pq.num_n_tiles = nout / kPksBN;
    CUtensorMap tq = tb;
    if (!dgrad) {  // 128 weight rows per CTA in one box (dgrad's map has 64-channel boxes)
      rc = make_weight_map(&tq, w, s.Cin, s.Cout, kPksBN / 2);
      if (rc) return rc;
    }
    rc = dgrad ? launch_igemm_pks<true>(ta, ta2, tq, pq, d, st) : launch_igemm_pks<false>(ta, ta2, tq, pq, d, st);
    if (rc != CONV3X3_ERR_UNSUPPORTED) return rc;  // (else the clusters do not fit: the tiles below)
  }
  // K split over two-CTA clusters (k_igemm_ks) where 128 x 256 tiles fill
  // between a quarter and all of the GPU's SMs in pairs and K is long: the
  // 8x8 layers with 1024 input channels.  Measured on GB300 (batch 64, 8x8):
  // 1024 -> 512 forward 41.3 -> 39.2 us against 128 x 128 one-CTA tiles, but
  // 512 -> 512 forward 25.4 -> 26.3 us (each CTA still streams 48 KB per
  // k-block, and the fill and the exchange weigh more at short K).
  // CONV3X3_KSPLIT=0|1 forces the choice (1 still needs a multiple of 256
  // output channels).
  const long long ks_tiles = (g.P() + BM - 1) / BM * ((nout + kKsBN - 1) / kKsBN);
  bool ks = !s2 && !ts.halo && pair_bn == 0 && nout % kKsBN == 0 && 2 * ks_tiles <= d.num_sms &&
            4 * ks_tiles >= d.num_sms && prm.kchunks >= 16;
  if (const char* e = std::getenv("CONV3X3_KSPLIT"))
    ks = std::strcmp(e, "0") != 0 && !s2 && !ts.halo && pair_bn == 0 && nout % kKsBN == 0;
  if (ks) {
    prm.num_m_tiles = (int)((g.P() + BM - 1) / BM);
    prm.num_n_tiles = nout / kKsBN;
    if (!dgrad) {  // one 256-row box per weight tile (dgrad's map has 64-row boxes)
      rc = make_weight_map(&tb, w, s.Cin, s.Cout, kKsBN);
      if (rc) return rc;
    }
    return dgrad ? launch_igemm_ks<true>(ta, ta2, tb, prm, d, st) : launch_igemm_ks<false>(ta, ta2, tb, prm, d, st);
  }
  if (pair_bn && !s2) {
    // a pair tile is 256 pixels (128 per CTA) x pair_bn channels, each CTA
    // loading pair_bn / 2 weight rows (as three 64-row boxes at 384)
    prm.num_m_tiles = (int)((g.P() + 2 * BM - 1) / (2 * BM));
    prm.num_n_tiles = (nout + pair_bn - 1) / pair_bn;
    // the weight boxes: pair_bn / 2 rows, and 64 rows for half-width items
    // (dgrad's map already has 64-channel boxes)
    CUtensorMap tb64 = tb;
    if (!dgrad) {
      rc = make_weight_map(&tb, w, s.Cin, s.Cout, pair_bn == 384 ? 64 : pair_bn / 2);
      if (rc) return rc;
      if (pair_bn == 256) {
        rc = make_weight_map(&tb64, w, s.Cin, s.Cout, 64);
        if (rc) return rc;
      } else {
        tb64 = tb;
      }
    }
#define C3_PAIR(BN_, KC_)                                                              \
  return dgrad ? launch_igemm_pair<true, BN_, KC_>(ta, ta2, tb, tb64, prm, d, st)      \
               : launch_igemm_pair<false, BN_, KC_>(ta, ta2, tb, tb64, prm, d, st)
    // two 64-channel chunks per stage where K is a whole number of them;
    // CONV3X3_PAIR_KC=1 keeps one
    int pkc = prm.kchunks % 2 == 0 ? 2 : 1;
    if (const char* e = std::getenv("CONV3X3_PAIR_KC"))
      if (std::strcmp(e, "1") == 0) pkc = 1;
    if (pair_bn == 128) {
      if (pkc == 2) C3_PAIR(128, 2);
      C3_PAIR(128, 1);
    }
    if (pair_bn == 192) C3_PAIR(192, 1);
    if (pair_bn == 384) C3_PAIR(384, 1);
    if (pkc == 2) C3_PAIR(256, 2);
    C3_PAIR(256, 1);
#undef C3_PAIR
  }
  // Two 64-channel chunks per k-block where the tile's MMAs are short (see
  // IgemmCfg); CONV3X3_KC=1|2 overrides the choice (tuning).
  int kc = (ts.mt == 1 && bn == 128) ? 2 : 1;
  if (const char* e = std::getenv("CONV3X3_KC")) {
    const int v = std::atoi(e);
    if (v == 1 || v == 2) kc = v;
  }
  if (kc == 2 && !((ts.mt == 1 && (bn == 128 || bn == 192 || bn == 256)) || (ts.mt == 2 && bn == 128)))
    kc = 1;
  prm.kgroups = (prm.kchunks + kc - 1) / kc;
#define C3_LAUNCH(BN_, MT_, KC_) \
  return dgrad ? launch_igemm<BN_, MT_, true, KC_>(ta, ta2, tb, prm, d, st) \
               : launch_igemm<BN_, MT_, false, KC_>(ta, ta2, tb, prm, d, st)
  if (kc == 2) {
    if (ts.mt == 2) C3_LAUNCH(128, 2, 2);
    if (bn == 128) C3_LAUNCH(128, 1, 2);
    if (bn == 192) C3_LAUNCH(192, 1, 2);
    C3_LAUNCH(256, 1, 2);
  }
  if (ts.mt == 2) {
    if (bn == 64) C3_LAUNCH(64, 2, 1);
    // (with z_in too: a warp's 2-byte z_in loads read one 64-byte run of 32
    // channels per pixel; measured on the 128-channel 64x64 layer's fused
    // dgrad: 118 us on the untransposed tile)
    if (trans && !s2)
      return dgrad ? launch_igemm<128, 2, true, 1, true>(ta, ta2, tb, prm, d, st)
                   : launch_igemm<128, 2, false, 1, true>(ta, ta2, tb, prm, d, st);
    C3_LAUNCH(128, 2, 1);
  }
  switch (bn) {
    case 64: C3_LAUNCH(64, 1, 1);
    case 128: C3_LAUNCH(128, 1, 1);
    case 192: C3_LAUNCH(192, 1, 1);
    default: C3_LAUNCH(256, 1, 1);
  }
#undef C3_LAUNCH
}

struct WgPlan {
  int num_mb, num_cb, tiles, kb_total, kb_per_split, S;
};

WgPlan wg_plan(const Shape& s) {
  WgPlan pl;
  pl.num_mb = (s.Cout + 127) / 128;
  pl.num_cb = (s.Cin + 127) / 128;
  pl.tiles = pl.num_mb * 3 * pl.num_cb;
  pl.kb_total = (int)((s.P() + kWgPix - 1) / kWgPix);
  // Cost in units of one 64-pixel k-block on one CTA, fitted to GB300 timings:
  // waves x (k-blocks per split + ~20 for a CTA's fill, drain and partial
  // write) + the partial-sum traffic, ~0.3 per MB of dw per split.
  const double dw_mb = (double)s.Cout * 9.0 * s.Cin * 4.0 / 1e6;
  double best = -1;
  int bestS = 1;
  for (int S = 1; S <= pl.kb_total && S <= 1024; ++S) {
    int per = (pl.kb_total + S - 1) / S;
    int Sreal = (pl.kb_total + per - 1) / per;
    if (Sreal != S) continue;
    long long units = (long long)pl.tiles * S;
    long long waves = (units + kPlanSms - 1) / kPlanSms;
    double cost = (double)waves * (per + 20) + 0.3 * S * dw_mb;
    if (best < 0 || cost < best) {
      best = cost;
      bestS = S;
    }
  }
  // CONV3X3_WGRAD_SPLITS=<S> overrides the split count (tuning); the workspace
  // size follows, so set it before querying the size.
  if (const char* e = std::getenv("CONV3X3_WGRAD_SPLITS")) {
    const int v = std::atoi(e);
    if (v >= 1 && v <= pl.kb_total) bestS = v;
  }
  pl.kb_per_split = (pl.kb_total + bestS - 1) / bestS;
  pl.S = (pl.kb_total + pl.kb_per_split - 1) / pl.kb_per_split;
  return pl;
}

// Two-CTA wgrad: Cout a multiple of 256 (pair tiles of 256 output channels).
bool wg_pair_shape(const Shape& s) { return s.Cout % 256 == 0; }

// Output channels [0, cpair) of a Cout above 256 that is not a multiple of
// 256 run as pair tiles, the rest [cpair, Cout) on one-CTA tiles, in two
// launches with a split plan each (one workspace, one reduction): 0 where
// that is not taken.  Each part pays its own fill, partial write and launch,
// so the hybrid is taken only where the one-CTA plan for all of Cout leaves
// over a quarter of the SMs idle.  Measured on GB300 (batch 64, 16x16):
// 768 -> 384 (108 of 152 SMs busy) 81 -> 69 us; 384 -> 384 (135 busy)
// 42 -> 56 us and 256 -> 384 (144 busy) 31 -> 46 us, so both keep one-CTA
// tiles.  CONV3X3_WGRAD_HYBRID=1 takes it wherever it applies, =0 nowhere.
int wg_hybrid_cpair(const Shape& g) {
  if (g.Cout <= 256 || wg_pair_shape(g)) return 0;
  int mode = -1;
  if (const char* e = std::getenv("CONV3X3_WGRAD_HYBRID")) mode = std::strcmp(e, "0") == 0 ? 0 : 1;
  if (mode == 0) return 0;
  if (mode < 0) {
    const WgPlan pl = wg_plan(g);
    if (4LL * pl.tiles * pl.S >= 3LL * kPlanSms) return 0;
  }
  return g.Cout / 256 * 256;
}


// Split plan of k_wgrad_pair: the same cost model over pair tiles and the
// kPlanSms / 2 cluster slots.
WgPlan wg_plan_pair(const Shape& s) {
  WgPlan pl;
  pl.num_mb = s.Cout / 256;
  pl.num_cb = (s.Cin + 127) / 128;
  pl.tiles = pl.num_mb * 3 * pl.num_cb;
  pl.kb_total = (int)((s.P() + kWgPix - 1) / kWgPix);
  const double dw_mb = (double)s.Cout * 9.0 * s.Cin * 4.0 / 1e6;
  const int slots = kPlanSms / 2;
  double best = -1;
  int bestS = 1;
  for (int S = 1; S <= pl.kb_total && S <= 1024; ++S) {
    int per = (pl.kb_total + S - 1) / S;
    int Sreal = (pl.kb_total + per - 1) / per;
    if (Sreal != S) continue;
    long long units = (long long)pl.tiles * S;
    long long waves = (units + slots - 1) / slots;
    double cost = (double)waves * (per + 20) + 0.3 * S * dw_mb;
    if (best < 0 || cost < best) {
      best = cost;
      bestS = S;
    }
  }
  if (const char* e = std::getenv("CONV3X3_WGRAD_SPLITS")) {
    const int v = std::atoi(e);
    if (v >= 1 && v <= pl.kb_total) bestS = v;
  }
  pl.kb_per_split = (pl.kb_total + bestS - 1) / bestS;
  pl.S = (pl.kb_total + pl.kb_per_split - 1) / pl.kb_per_split;
  return pl;
}

// The two parts of a hybrid weight gradient (wg_hybrid_cpair): the pair plan
// over output channels [0, cpair), the one-CTA plan over [cpair, Cout), and
// the slices of their shared workspace (the larger split count).
struct WgHybrid {
  int cpair;
  WgPlan pp, ps;
  int Sreg;
};

WgHybrid wg_plan_hybrid(const Shape& g) {
  WgHybrid h;
  h.cpair = wg_hybrid_cpair(g);
  Shape gp = g, gs = g;
  gp.Cout = h.cpair;
  gs.Cout = g.Cout - h.cpair;
  h.pp = wg_plan_pair(gp);
  h.ps = wg_plan(gs);
  h.Sreg = h.pp.S > h.ps.S ? h.pp.S : h.ps.S;
  return h;
}

}  // namespace

bool tc_supported(int pass, const Shape& s) {
  (void)pass;
  // im2col corner offsets and coordinates are 16/32-bit; the kernels index pixels with int.
  if (s.P() >= (1LL << 31)) return false;
  if (s.H > 65535 || s.W > 65535) return false;
  // stride 2: TMA boxes of 64 channels over tensors at least that wide
  if (s.u != 1 && (s.u != 2 || s.Cin < BKC || s.Cout < BKC)) return false;
  return true;
}

// A channel split runs on the tensor cores when the first part is a whole
// number of 64-channel K chunks (every TMA box then lies in one part).
bool tc_supports_cat(const Shape& s, const CatSplit& cat) {
  return !cat.on() || (cat.Ca % BKC == 0 && cat.Ca > 0 && cat.Ca < s.Cin);
}

int tc_fwd(const void* x, const void* w, const float* bias, void* y, const Shape& s, int act,
           int out_f32, const EpiExtra& ex, const CatSplit& cat, const DevCtx& d,
           cudaStream_t st) {
  if (!tc_supports_cat(s, cat)) return CONV3X3_ERR_UNSUPPORTED;
  if (s.Cin == 8 && s.Cout <= 256 && !cat.on() && s.u == 1)
    return run_stem_fwd(x, w, bias, y, s, act, out_f32, ex, d, st);
  return run_igemm(false, x, s.Cin, w, bias, y, s, act, out_f32, ex, cat, d, st);
}

int tc_dgrad(const void* dy, const void* w, void* dx, const Shape& s, int out_f32,
             const EpiExtra& ex, const CatSplit& cat, const DevCtx& d, cudaStream_t st) {
  if (!tc_supports_cat(s, cat)) return CONV3X3_ERR_UNSUPPORTED;
  // a forced im2col tile (CONV3X3_TILE) keeps the 8-channel dgrad on k_igemm
  if (!cat.on() && stem_dgrad_fits(s) && std::getenv("CONV3X3_TILE") == nullptr)
    return run_stem_dgrad(dy, w, dx, s, out_f32, ex, d, st);
  return run_igemm(true, dy, s.Cout, w, nullptr, dx, s, CONV3X3_ACT_NONE, out_f32, ex, cat, d, st);
}

// Cin == 8: one tile per 128 output channels; splits fill the GPU once.
WgPlan wg_plan_c8(const Shape& s) {
  WgPlan pl;
  pl.num_mb = (s.Cout + 127) / 128;
  pl.num_cb = 1;
  pl.tiles = pl.num_mb;
  pl.kb_total = (int)((s.P() + kWgPix - 1) / kWgPix);
  int S = kPlanSms / pl.tiles;
  if (S < 1) S = 1;
  if (S > pl.kb_total) S = pl.kb_total;
  pl.kb_per_split = (pl.kb_total + S - 1) / S;
  pl.S = (pl.kb_total + pl.kb_per_split - 1) / pl.kb_per_split;
  return pl;
}

// Image width for the row-shifted x layout of k_wgrad, or 0 for im2col: stride
// 1, a width of 16, 32 or 64 and images of a whole number of 64-pixel
// k-blocks (every k-block is whole image rows of one image).  By default only
// width 64 takes it: measured on GB300 (CUDA events, batch 64) it ran the
// 128-channel 64x64 layer in 68 instead of 72 us, while at widths 32 and 16 --
// two and four image rows per k-block, three MMAs per K step where im2col
// needs two -- it ran 3-12 % slower.  CONV3X3_WGRAD_ROWS=0 forces im2col,
// =1 the row-shifted layout wherever it applies (tuning and tests).
int wg_row_width(const Shape& s) {
  int mode = -1;
  if (const char* e = std::getenv("CONV3X3_WGRAD_ROWS")) mode = std::strcmp(e, "0") == 0 ? 0 : 1;
  if (mode == 0 || s.u != 1 || !(s.W == 16 || s.W == 32 || s.W == 64)) return 0;
  if (mode < 0 && s.W != 64) return 0;
  return ((long long)s.H * s.W) % kWgPix == 0 ? s.W : 0;
}

// The split plan runs over dy's pixel grid.
Shape wg_grid(const Shape& s) {
  Shape g = s;
  g.H = s.Ho();
  g.W = s.Wo();
  g.u = 1;
  return g;
}

size_t tc_wgrad_workspace(const Shape& s, int /*num_sms*/) {
  if (s.Cin == 8 && s.u == 1) {
    WgPlan pl = wg_plan_c8(s);
    return (size_t)pl.S * (size_t)((long long)s.Cout * 72 + s.Cout) * sizeof(float);
  }
  const Shape g = wg_grid(s);
  int S = wg_plan(g).S;
  // room for either kernel's splits, whichever the call takes
  if (wg_pair_shape(g)) {
    const int Sp = wg_plan_pair(g).S;
    if (Sp > S) S = Sp;
  }
  if (wg_hybrid_cpair(g)) {
    const WgHybrid h = wg_plan_hybrid(g);
    if (h.Sreg > S) S = h.Sreg;
  }
  long long dwsize = (long long)s.Cout * 9 * s.Cin;
  return (size_t)S * (size_t)(dwsize + s.Cout) * sizeof(float);
}

int run_wgrad_c8(const void* x, const void* dy, float* dw, float* db, const Shape& s, void* ws,
                 const DevCtx& d, cudaStream_t st) {
  WgPlan pl = wg_plan_c8(s);
  // width 64 (each 64-pixel k-block is one image row): x staged as three
  // column-shifted copies of three halo rows, six 3-row boxes per k-block;
  // otherwise (or with CONV3X3_STEM_ROWS=0) as nine im2col boxes.  Measured
  // on the 64x64 batch-64 stem (call, L2 flushed): 43 us with im2col boxes,
  // 33.3 us with two 512-byte row boxes per tap, 28.7 us with one box of
  // three pixel-pair rows and three N = 32 MMAs per K step.
  bool halo = s.W == 64;
  if (const char* e = std::getenv("CONV3X3_STEM_ROWS"))
    if (std::strcmp(e, "0") == 0) halo = false;
  CUtensorMap tdy, tx;
  int rc = make_rows_map(&tdy, dy, s.P(), s.Cout);
  if (rc) return rc;
  rc = halo ? make_row_map(&tx, x, s.N, s.H, s.W, 256, 3)
            : make_im2col_map(&tx, x, s.N, s.H, s.W, 8, kWgPix, 8, false);
  if (rc) return rc;
  WgradParams prm;
  prm.part = static_cast<float*>(ws);
  prm.P = (int)s.P();
  prm.H = s.H;
  prm.W = s.W;
  prm.Cin = s.Cin;
  prm.Cout = s.Cout;
  prm.ca = s.Cin;
  prm.ustride = 1;
  prm.kb_total = pl.kb_total;
  prm.kb_per_split = pl.kb_per_split;
  prm.S = pl.S;
  prm.num_mb = pl.num_mb;
  prm.num_cb = 1;
  prm.status = d.status;
  prm.wait_ns = d.wait_ns;
  if (halo) {
    // the partials [S][Cout][72] fp32 as a 3-D map for TMA stores: box {72, 32
    // channels, 1 split} (CONV3X3_WGRAD_PART_TMA=0 keeps per-thread stores)
    CUtensorMap tpart = tdy;  // (unused unless part_tma)
    prm.part_tma = 0;
    const char* pe = std::getenv("CONV3X3_WGRAD_PART_TMA");
    if (!(pe && std::strcmp(pe, "0") == 0)) {
      PFN_encodeTiled enc = encode_tiled_fn();
      cuuint64_t dims[3] = {72, (cuuint64_t)s.Cout, (cuuint64_t)pl.S};
      cuuint64_t strides[2] = {288, (cuuint64_t)s.Cout * 288};
      cuuint32_t box[3] = {72, 32, 1};
      cuuint32_t estr[3] = {1, 1, 1};
      if (enc && enc(&tpart, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, prm.part, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
        prm.part_tma = 1;
    }
    if (set_smem(k_wgrad_c8h, kWhSmem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
    launch_pdl(k_wgrad_c8h, dim3(pl.tiles * pl.S), dim3(kThreads), kWhSmem, st, tdy, tx, tpart, prm);
  } else {
    if (set_smem(k_wgrad_c8, kWc8Smem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
    launch_pdl(k_wgrad_c8, dim3(pl.tiles * pl.S), dim3(kThreads), kWc8Smem, st, tdy, tx, prm);
  }
  if (cudaGetLastError() != cudaSuccess) return CONV3X3_ERR_CUDA;
  return launch_wgrad_reduce(prm.part, dw, db, (long long)s.Cout * 72, s.Cout, pl.S, pl.S, st);
}

// The wgrad partials part [S][Cout][9][Cin] fp32 as a 4-D map for TMA stores:
// box {32 channels, 1 tap, 32 output channels, 1 split}, 128-byte swizzle
// (the staging layout of wg_store_partials).  Taken for Cin >= 32 (a box
// narrower than its tensor); CONV3X3_WGRAD_PART_TMA=0 keeps per-thread stores.
bool make_part_map(CUtensorMap* m, float* part, int Cin, int Cout, int S) {
  if (Cin < 32) return false;
  if (const char* e = std::getenv("CONV3X3_WGRAD_PART_TMA"))
    if (std::strcmp(e, "0") == 0) return false;
  PFN_encodeTiled enc = encode_tiled_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)Cin, 9, (cuuint64_t)Cout, (cuuint64_t)S};
  cuuint64_t strides[3] = {(cuuint64_t)Cin * 4, (cuuint64_t)Cin * 36, (cuuint64_t)Cout * Cin * 36};
  cuuint32_t box[4] = {32, 1, 32, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, part, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_wgrad(const void* x, const void* dy, float* dw, float* db, const Shape& s, void* ws,
             size_t ws_bytes, const CatSplit& cat, const DevCtx& d, cudaStream_t st) {
  if (!tc_supports_cat(s, cat)) return CONV3X3_ERR_UNSUPPORTED;
  if (ws == nullptr || ws_bytes < tc_wgrad_workspace(s, d.num_sms)) return CONV3X3_ERR_WORKSPACE;
  if (s.Cin == 8 && !cat.on() && s.u == 1) return run_wgrad_c8(x, dy, dw, db, s, ws, d, st);
  const Shape g = wg_grid(s);
  WgPlan pl = wg_plan(g);
  CUtensorMap tdy, tx, tx2;
  int rc = make_rows_map(&tdy, dy, g.P(), s.Cout);
  if (rc) return rc;
  rc = make_im2col_map(&tx, x, s.N, s.H, s.W, cat.on() ? cat.Ca : s.Cin, kWgPix, BKC, true, s.u);
  if (rc) return rc;
  if (cat.on()) {
    rc = make_im2col_map(&tx2, cat.b, s.N, s.H, s.W, s.Cin - cat.Ca, kWgPix, BKC, true, s.u);
    if (rc) return rc;
  } else {
    tx2 = tx;
  }
  WgradParams prm;
  prm.part = static_cast<float*>(ws);
  prm.P = (int)g.P();
  prm.H = g.H;
  prm.W = g.W;
  prm.Cin = s.Cin;
  prm.Cout = s.Cout;
  prm.ca = cat.on() ? cat.Ca : s.Cin;
  prm.ustride = s.u;
  prm.kb_total = pl.kb_total;
  prm.kb_per_split = pl.kb_per_split;
  prm.S = pl.S;
  prm.num_mb = pl.num_mb;
  prm.num_cb = pl.num_cb;
  prm.status = d.status;
  prm.wait_ns = d.wait_ns;
  const int hw = wg_row_width(s);
  // Two-CTA tiles for Cout a multiple of 256 with im2col x;
  // CONV3X3_WGRAD_PAIR=0 keeps the one-CTA kernel, =1 is the default.
  bool pair_ok = true;
  if (const char* e = std::getenv("CONV3X3_WGRAD_PAIR"))
    if (std::strcmp(e, "0") == 0) pair_ok = false;
  const bool pair = hw == 0 && pair_ok && wg_pair_shape(g);
  if (pair) {
    const WgPlan pp = wg_plan_pair(g);
    prm.kb_total = pp.kb_total;
    prm.kb_per_split = pp.kb_per_split;
    prm.S = pp.S;
    prm.num_mb = pp.num_mb;  // 256-channel pair blocks
    prm.num_cb = pp.num_cb;
    CUtensorMap tpart = tdy;  // (unused unless part_tma)
    prm.part_tma = make_part_map(&tpart, prm.part, s.Cin, s.Cout, pp.S) ? 1 : 0;
    if (set_smem(k_wgrad_pair, kWpSmem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
    launch_pdl(k_wgrad_pair, dim3(2 * pp.tiles * pp.S), dim3(kThreads), kWpSmem, st, tdy, tx, tx2, tpart,
               prm);
    if (cudaGetLastError() != cudaSuccess) return CONV3X3_ERR_CUDA;
    return launch_wgrad_reduce(prm.part, dw, db, (long long)s.Cout * 9 * s.Cin, s.Cout, pp.S, pp.S, st);
  }
  const int cpair = (hw == 0 && pair_ok) ? wg_hybrid_cpair(g) : 0;
  if (cpair) {
    // pair tiles over output channels [0, cpair), then one-CTA tiles over
    // [cpair, Cout); both write the shared workspace (Sreg slices), and the
    // reduction sums each part's own splits
    const WgHybrid h = wg_plan_hybrid(g);
    CUtensorMap tpart = tdy;  // (unused unless part_tma)
    const int part_tma = make_part_map(&tpart, prm.part, s.Cin, s.Cout, h.Sreg) ? 1 : 0;
    WgradParams pa = prm;
    pa.kb_total = h.pp.kb_total;
    pa.kb_per_split = h.pp.kb_per_split;
    pa.S = h.Sreg;
    pa.num_mb = h.pp.num_mb;
    pa.num_cb = h.pp.num_cb;
    pa.part_tma = part_tma;
    if (set_smem(k_wgrad_pair, kWpSmem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
    launch_pdl(k_wgrad_pair, dim3(2 * h.pp.tiles * h.pp.S), dim3(kThreads), kWpSmem, st, tdy, tx, tx2, tpart,
               pa);
    if (cudaGetLastError() != cudaSuccess) return CONV3X3_ERR_CUDA;
    WgradParams pb = prm;
    pb.kb_total = h.ps.kb_total;
    pb.kb_per_split = h.ps.kb_per_split;
    pb.S = h.Sreg;
    pb.num_mb = h.ps.num_mb;
    pb.num_cb = h.ps.num_cb;
    pb.mb0 = cpair / 128;
    pb.part_tma = part_tma;
    if (set_smem(k_wgrad<0>, WgCfg<0>::kSmem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;
    launch_pdl(k_wgrad<0>, dim3(h.ps.tiles * h.ps.S), dim3(kThreads), WgCfg<0>::kSmem, st, tdy, tx, tx2, tpart,
               pb);
    if (cudaGetLastError() != cudaSuccess) return CONV3X3_ERR_CUDA;
    return launch_wgrad_reduce2(prm.part, dw, db, (long long)s.Cout * 9 * s.Cin, s.Cout, h.Sreg, h.pp.S, h.ps.S,
                                cpair, st);
  }
  if (hw) {
    // row-shifted x: per image row one box of (W + 2) pixels x 64 channels
    rc = make_halo_map(&tx, x, s.N, s.H, s.W, cat.on() ? cat.Ca : s.Cin, 1, s.W + 2);
    if (rc) return rc;
    if (cat.on()) {
      rc = make_halo_map(&tx2, cat.b, s.N, s.H, s.W, s.Cin - cat.Ca, 1, s.W + 2);
      if (rc) return rc;
    } else {
      tx2 = tx;
    }
  }
  CUtensorMap tpart = tdy;  // (unused unless part_tma)
  prm.part_tma = make_part_map(&tpart, prm.part, s.Cin, s.Cout, pl.S) ? 1 : 0;
#define C3_WG(HW_)                                                                               \
  do {                                                                                           \
    using Cfg = WgCfg<HW_>;                                                                      \
    if (set_smem(k_wgrad<HW_>, Cfg::kSmem, d.device) != CONV3X3_OK) return CONV3X3_ERR_CUDA;     \
    launch_pdl(k_wgrad<HW_>, dim3(pl.tiles * pl.S), dim3(kThreads), Cfg::kSmem, st, tdy, tx, tx2, \
               tpart, prm);                                                                      \
  } while (0)
  if (hw == 64)
    C3_WG(64);
  else if (hw == 32)
    C3_WG(32);
  else if (hw == 16)
    C3_WG(16);
  else
    C3_WG(0);
#undef C3_WG
  if (cudaGetLastError() != cudaSuccess) return CONV3X3_ERR_CUDA;
  return launch_wgrad_reduce(prm.part, dw, db, (long long)s.Cout * 9 * s.Cin, s.Cout, pl.S, pl.S, st);
}

}  // namespace c3
