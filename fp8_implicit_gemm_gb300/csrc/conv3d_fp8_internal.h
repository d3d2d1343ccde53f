// conv3d_fp8_internal.h -- what the host launcher and the kernels of the library share.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace c3d {

constexpr int kBlockM = 128;        // rows (output positions) per tile = TMEM lanes
constexpr int kBlockK = 128;        // K_gemm bytes per pipeline stage (= one 128-byte swizzle row)
constexpr int kMmaK = 32;           // K of one tcgen05.mma kind::f8f6f4
constexpr int kATileBytes = kBlockM * kBlockK;  // 16 KB
constexpr int kNumThreads = 320;    // 4 epilogue warps, 4 A-loader warps, 1 TMA warp, 1 MMA warp
constexpr int kSmemBudget = 200 * 1024;
constexpr long long kSmemPerSm = 228 * 1024;    // shared memory of one SM
constexpr long long kPackLightSmem = 16384;     // one stage of the light pack's ring
constexpr int kMaxStages = 8;
constexpr int kEpiStageBytes = 2 * 32 * kBlockM * 2;  // two bf16 boxes [32 columns][128 rows]

// How the A operand (im2col rows of x) reaches shared memory.
enum : int {
  kRouteGather = 0,  // 16-byte cp.async gathers from a zero-padded channels-last copy of x
  kRouteIm2col = 1,  // TMA im2col loads from an unpadded channels-last copy (C % 32 == 0)
  kRouteGrid = 2,    // stride 1: M indexes the zero-padded grid of the input, so every tap is a
                     // shift along that grid; one TMA load of 128 + S - 1 grid positions feeds
                     // the S taps along W (CTA pairs only)
  kRouteDirect = 3,  // K_gemm in the caller's KCTRS order (channel outer, tap inner): B by TMA
                     // tiles of the caller's weights (no re-layout), A by TMA tiles of an
                     // explicit im2col of x that the pre-pass writes (one CTA; for layers with
                     // few output positions, whose weights are the bulk of the bytes)
};

// Source types of the quantiser (and of x when a run quantises it in the pack).
enum : int { kSrcE4m3 = 0, kSrcF32 = 1, kSrcBf16 = 2 };

// Status-word bits recorded by kernels whose bounded waits ran out.
enum : int {
  kStatusWaitFull = 1 << 0,       // MMA warp waiting for operands
  kStatusWaitEmpty = 1 << 1,      // a loader waiting for a free stage
  kStatusWaitAccFull = 1 << 2,    // epilogue waiting for an accumulator
  kStatusWaitAccEmpty = 1 << 3,   // MMA warp waiting for the epilogue to drain TMEM
  kStatusWaitDrain = 1 << 4,      // final drain of outstanding MMAs
};

struct ConvParams {
  // problem
  int N, C, D, H, W, K, T, R, S;  // C: bytes of one pixel's channels (channels * elem_bytes)
  int elem_bytes;        // 1: e4m3 inputs (kind::f8f6f4); 2: bfloat16 inputs (kind::f16)
  int sd, sh, sw, pd, ph, pw;
  int Do, Ho, Wo;
  int route;             // kRouteGather, kRouteIm2col, kRouteGrid or kRouteDirect (how A, and on
                         // the direct route B, reach shared memory)
  int a_cb;              // im2col route: channels per A sub-tile (32, 64 or 128 = its row bytes)
  int pk_pd, pk_ph, pk_pw;  // zero halo of the packed channels-last x (gather route only)
  int Dp, Hp, Wp;        // extents of the packed channels-last copy of x (halo included)
  int Dg, Hg, Wg;        // padded-grid route: extents of the zero-padded grid, D + 2 pd, ...
  int x_cl;              // the caller's x is channels-last (NDHWC): no transpose in the pack
  int epi_tma;           // whole tiles leave through TMA stores bounded by the map of y (output-
                         // position routes); otherwise explicit guarded stores
  int halo_once;         // the plan zeroed its padded copy at creation: the pack skips the halo
  int x_src_type;        // kSrcE4m3: x is e4m3 bytes; kSrcF32 / kSrcBf16: the pack quantises x
                         // (NCDHW values) with the device scale *scale_x
  int a_grid_im2col;     // padded-grid route: A by im2col loads from an unpadded channels-last x
                         // (the caller's); otherwise by 2D tiles of the zero-padded copy
  int dhw;               // Do*Ho*Wo
  int tiles_per_image;   // padded-grid route: M tiles per image (grid rows of d < Do planes)
  int npq;               // N*dhw, the M of the GEMM view
  int taps;              // T*R*S
  int kg;                // taps*C, the K of the GEMM view
  // tiling
  int pair;              // 1: CTA-pair kernel (cta_group::2, block_m = 256); 0: one-CTA kernel
  int block_m;           // M tile: 128 (one CTA) or 256 (CTA pair)
  int block_n;           // N tile (multiple of 32, <= 256)
  int m_tiles, n_tiles, k_blocks, splits, kb_per_split, num_units;
  int unit_base;         // this launch runs units unit_base .. unit_base + num_units - 1 (a plan
                         // that overlaps its pack with the GEMM runs the units in two launches)
  int full_tiles;        // tiles 0..full_tiles-1 are computed whole (one unit each, bf16 out);
                         // the others are split `splits` ways along K into fp32 partials
  int stages;
  int tmem_cols;         // allocated TMEM columns (power of two)
  int acc_stride;        // TMEM column offset between the two accumulator buffers
  // tensors
  const uint8_t* x;      // e4m3 NCDHW, or NDHWC when x_cl (caller's)
  const uint8_t* w;      // e4m3 KCTRS (caller's)
  uint8_t* xp;           // e4m3 [N][Dp][Hp][Wp][C], zero halo (workspace; null when the TMA
                         // routes read a channels-last x of the caller directly). Direct route:
                         // the explicit A = im2col(x), [npq][kg] bytes in (channel, tap) order
  uint8_t* wp;           // e4m3 [K][taps][C] (workspace)
  uint16_t* y;           // bf16 NCDHW (caller's)
  const float* scale_x;
  const float* scale_w;
  float* partials;       // fp32 [tile - full_tiles][split][block_n][block_m] (workspace)
  int* status;           // status word (workspace)
  uint32_t* write_count; // a library built with C3D_COUNT_WRITES (tests): one counter per output
                         // element, incremented by every store to it; null otherwise
  unsigned long long timeout_ns;
  int debug_flags;
};

// Launchers (defined in the .cu files). Each returns the CUDA error of its launch.
cudaError_t launch_pack(const ConvParams& p, cudaStream_t stream);
// The tiled transpose of x (e4m3 or bfloat16 NCDHW, W % 4 == 0, D*H*W*bytes % 16 == 0,
// C % 64 == 0: pack_transposes_x) over the positions [q_lo, q_hi) of every image's volume (q_lo a
// multiple of kPackTilePositions), with the weights and the remaining items when `whole` is set.
// `light`: one block an SM with a single 16 KB stage, small enough to run beside a GEMM CTA.
bool pack_transposes_x(const ConvParams& p);
constexpr int kPackTilePositions = 256;  // every tile length of the transposes divides it
cudaError_t launch_pack_range(const ConvParams& p, long long q_lo, long long q_hi, bool whole,
                              bool light, cudaStream_t stream);
cudaError_t launch_conv(const ConvParams& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                        const CUtensorMap& ymap, bool row_chk, int grid, cudaStream_t stream);
cudaError_t launch_splitk_reduce(const ConvParams& p, bool row_chk, cudaStream_t stream);
// quantiser (quant.cu): amax of |src| into *amax_bits (zeroed first); e4m3 codes of src with the
// scale of that amax; the scale itself into scale_out (and scale_copy when not null)
cudaError_t launch_amax(const void* src, int type, long long n, unsigned* amax_bits,
                        cudaStream_t stream);
cudaError_t launch_quant_cast(const void* src, int type, long long n, uint8_t* dst,
                              const unsigned* amax_bits, cudaStream_t stream);
cudaError_t launch_quant_finalize(const unsigned* amax_bits, float* scale_out, float* scale_copy,
                                  cudaStream_t stream);
size_t conv_smem_bytes(int block_n, int stages, bool epi_tma);
cudaError_t conv_set_smem_attr(size_t smem_bytes);  // both kernels
cudaError_t launch_conv_pair(const ConvParams& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                             const CUtensorMap& ymap, bool row_chk, int grid, cudaStream_t stream);
size_t conv_pair_smem_bytes(const ConvParams& p);
cudaError_t conv_pair_set_smem_attr(size_t smem_bytes);
int conv_pair_max_active_clusters(const ConvParams& p);  // 0 if the query fails

}  // namespace c3d
