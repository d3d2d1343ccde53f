// pack.cu -- operand re-layout in front of the implicit GEMM, and the split-K reduction behind it.
//
// The GEMM view orders K_gemm as (tap, channel) with the channel innermost, so that one row of the
// A tile for one tap is C contiguous bytes of one input pixel. The caller's x is NCDHW (channel
// outermost), so it is copied once per run into a channels-last buffer. For the TMA im2col route
// the copy is plain NDHWC (the TMA unit zero-fills taps outside the volume); for the cp.async
// gather route it carries an explicit zero halo of `pad` pixels on every spatial side, so that an
// A-tile row needs no bounds test, only the padded-row test (row < npq). The weights are re-laid
// from KCTRS to K x taps x C to match.
#include <algorithm>

#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "pack_items.cuh"
#include "quant.cuh"

namespace c3d {

// Blocks [0, item_blocks) run the items in a grid-stride loop; the blocks after them one weight
// tile each (pack_w_tile, kWTileBytes of dynamic shared memory).
__global__ void __launch_bounds__(256) pack_kernel(ConvParams p, PackPlan q, int item_blocks) {
  pdl_launch_dependents();  // the implicit GEMM may start its prologue while the pack runs
  extern __shared__ __align__(16) uint8_t wsm[];
  if ((int)blockIdx.x >= item_blocks) {
    pack_w_tile(p, q, (long long)blockIdx.x - item_blocks, wsm);
    return;
  }
  const PackCtx c = pack_ctx(p, q);
  const long long total = c.e3 + q.w_items;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)item_blocks * blockDim.x)
    pack_item(p, q, c, g);
}

// Tiled transpose of the interior of an NCDHW x into the e4m3 channels-last copy, quantising
// fp32 / bfloat16 values (kType) on the way. A tile is kTileP consecutive positions of one image's
// D x H x W volume and kCT channels. The first tile_blocks blocks walk the tiles blockIdx.x,
// + tile_blocks, ... through two shared-memory stages (one tile each when tile_blocks == x_tiles):
//   1. the kCT source rows of the next tile (each kTileP contiguous elements of one channel plane)
//      go into the free stage with 16-byte cp.async copies, in flight while
//   2. each thread takes one (position, 16-channel chunk) of the current tile: it reads the 16
//      values of its column (consecutive threads read consecutive positions: no bank conflicts),
//      quantises them and stores the 16 codes with one 16-byte store into the padded
//      channels-last copy.
// The source is read in runs of kTileP elements per channel plane (1.5 KB from fp32). The item path
// it replaced (one thread = 16 channels x 4 pixels, 16 planes per thread) made the quantised step
// of the large layer 450 us (fp32 x) and 409 us (bf16 x).
// Blocks past the persistent ones run the remaining items (halo, weights by items) of the item
// path, then one weight tile each (pack_w_tile).
template <int kType>
__host__ __device__ constexpr int src_bytes() {
  return kType == kSrcF32 ? 4 : 2;  // fp32 or bfloat16
}
// Positions of a tile and blocks an SM: an fp32 x takes tiles of 384 positions, one per block, 4
// blocks an SM (48 KB each, <= 64 registers a thread: the large layer's pack 73.9 -> 69.8 us
// against 512 positions and 3 blocks); a bfloat16 x keeps 512 positions and 3 persistent blocks
// with two 32 KB stages (<= 80 registers), which measured faster for it (60.2-63.3 against
// 64.6 us with 384 positions and 4 blocks).
template <int kType>
__host__ __device__ constexpr int tile_positions() {
  return kType == kSrcF32 ? 384 : 512;
}
template <int kType>
__host__ __device__ constexpr int tiled_blocks_per_sm() {
  return kType == kSrcF32 ? 4 : 3;
}

template <int kType, int kCT>
__global__ void __launch_bounds__(256, tiled_blocks_per_sm<kType>()) pack_x_tiled_kernel(
    ConvParams p, PackPlan q, long long x_tiles, int tile_blocks, long long rest_blocks) {
  pdl_launch_dependents();  // the implicit GEMM may start its prologue while the pack runs
  constexpr int kTileP = tile_positions<kType>();
  constexpr int kEB = src_bytes<kType>();
  constexpr int kRowBytes = kTileP * kEB;
  constexpr int kStageBytes = kCT * kRowBytes;
  extern __shared__ __align__(16) uint8_t raw[];  // [2][kCT][kTileP] source elements
  const long long b = blockIdx.x;
  if (b >= tile_blocks + rest_blocks) {
    pack_w_tile(p, q, b - tile_blocks - rest_blocks, raw);  // the stages hold kWTileBytes
    return;
  }
  if (b >= tile_blocks) {
    const PackCtx c = pack_ctx(p, q);
    const long long total = c.e3 + q.w_items;
    const long long stride = rest_blocks * blockDim.x;
    for (long long g = c.e1 + (b - tile_blocks) * blockDim.x + threadIdx.x; g < total; g += stride)
      pack_rest_item(p, q, c, g);
    return;
  }
  const long long dhw = (long long)p.D * p.H * p.W;
  const long long pt = (dhw + kTileP - 1) / kTileP;
  const int ctn = p.C / kCT;
  // every row starts 16-byte aligned, and vectors never straddle dhw: cp.async copies
  const bool vec = (dhw * kEB) % 16 == 0;
  const float qs = __ldg(p.scale_x);
  struct Tile {
    int n, c0, valid;
    long long q0;
    const uint8_t* src;
  };
  auto tile_at = [&](long long t) {  // position tiles fastest, then channel groups, then images
    Tile tl;
    const long long pi = t % pt, rest = t / pt;
    tl.n = (int)(rest / ctn);
    tl.c0 = (int)(rest % ctn) * kCT;
    tl.q0 = pi * kTileP;
    tl.valid = dhw - tl.q0 < kTileP ? (int)(dhw - tl.q0) : kTileP;
    tl.src = p.x + (((long long)tl.n * p.C + tl.c0) * dhw + tl.q0) * kEB;
    return tl;
  };
  auto issue = [&](const Tile& tl, uint8_t* stage) {  // cp.async copies of a tile, no wait
    constexpr int kVecs = kRowBytes / 16;
    constexpr int kIters = kCT * kVecs / 256;  // blockDim.x == 256
    const int vec_valid = (tl.valid * kEB + 15) / 16;
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
      const int t = threadIdx.x + 256 * i;
      const int r = t / kVecs, c = t - r * kVecs;
      if (c < vec_valid)
        cp_async_16_zfill(smem_u32(stage + r * kRowBytes + c * 16),
                          tl.src + (long long)r * dhw * kEB + (long long)c * 16, 16);
    }
  };
  int sidx = 0;
  if (vec) issue(tile_at(b), raw);
  cp_async_commit();
  for (long long t = b; t < x_tiles; t += tile_blocks) {
    const Tile tl = tile_at(t);
    uint8_t* stage = raw + sidx * kStageBytes;
    const long long nt = t + tile_blocks;
    if (vec && nt < x_tiles) issue(tile_at(nt), raw + (sidx ^ 1) * kStageBytes);
    cp_async_commit();
    if (vec) {
      cp_async_wait_group<1>();  // this thread's copies of tile t have landed
    } else {
      for (int i = threadIdx.x; i < kCT * kTileP; i += blockDim.x) {
        const int r = i / kTileP, e = i - r * kTileP;
        if (e < tl.valid) {
          const uint8_t* a = tl.src + ((long long)r * dhw + e) * kEB;
          uint8_t* o = stage + r * kRowBytes + e * kEB;
          if (kEB == 4)
            *reinterpret_cast<uint32_t*>(o) = __ldg(reinterpret_cast<const uint32_t*>(a));
          else
            *reinterpret_cast<uint16_t*>(o) = __ldg(reinterpret_cast<const uint16_t*>(a));
        }
      }
    }
    __syncthreads();
    constexpr int kChunks = kCT / 16;
    for (int i = threadIdx.x; i < kTileP * kChunks; i += blockDim.x) {
      const int k = i / kTileP, e = i - k * kTileP;  // positions fastest across threads
      if (e >= tl.valid) continue;
      uint32_t w[4];
#pragma unroll
      for (int j4 = 0; j4 < 4; ++j4) {
        const int r = 16 * k + 4 * j4;
        float v[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          if (kType == kSrcF32)
            v[m] = *reinterpret_cast<const float*>(stage + (r + m) * kRowBytes + 4 * e);
          else
            v[m] = __uint_as_float(
                (uint32_t)*reinterpret_cast<const uint16_t*>(stage + (r + m) * kRowBytes + 2 * e)
                << 16);
        }
        w[j4] = quant4(v[0], v[1], v[2], v[3], qs);
      }
      const long long qq = tl.q0 + e;  // position within the image's volume -> (d, h, w)
      const int wq = (int)(qq % p.W);
      const long long dh = qq / p.W;
      const int hq = (int)(dh % p.H), dq = (int)(dh / p.H);
      uint8_t* dst = p.xp + ((((long long)tl.n * p.Dp + dq + p.pk_pd) * p.Hp + hq + p.pk_ph) *
                                 p.Wp + wq + p.pk_pw) * p.C + tl.c0 + 16 * k;
      *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();  // the stage is free for the copies two tiles on
    sidx ^= 1;
  }
  cp_async_wait_all();
}

// tile_blocks == x_tiles: one tile per block, no prefetch, so one stage of shared memory is enough
template <int kType, int kCT>
static cudaError_t launch_tiled_ct(const ConvParams& p, const PackPlan& q, long long x_tiles,
                                   long long tile_blocks, long long rest_blocks,
                                   cudaStream_t stream) {
  constexpr size_t stage = (size_t)kCT * tile_positions<kType>() * src_bytes<kType>();
  static_assert(stage >= (size_t)kWTileBytes, "the weight tiles use the stages");
  const size_t smem = tile_blocks < x_tiles ? 2 * stage : stage;
  const unsigned blocks = (unsigned)(tile_blocks + rest_blocks + q.w_blocks);
  auto k = pack_x_tiled_kernel<kType, kCT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<blocks, 256, smem, stream>>>(p, q, x_tiles, (int)tile_blocks, rest_blocks);
  return cudaGetLastError();
}

// The ring of the tiled packs. An x tile is kCG channels x kTP consecutive positions of one
// image's D x H x W volume, 16 KB: kCG runs of kTP source elements (kEB bytes each), one per
// channel plane. Every block walks the tiles blockIdx.x, + gridDim.x, ... -- the x tiles, then the
// weight tiles (pack_w_tile) -- through kRingStages shared-memory stages: the runs of the x tile
// two steps ahead arrive by 16-byte cp.async copies (a warp's 32 copies are whole 128-byte lines
// of the source) while tile_fn turns the current stage into 16-byte chunks of the channels-last
// copy. Row r of a stage keeps its 16-byte chunks rotated by (r / kRotRows) * kRotB bytes, which
// tile_fn's reads undo (each kernel picks kRotRows and kRotB so that the words its warps read
// fall in distinct banks). Then the blocks share the remaining items (halo chunks, weights by
// items) in a grid-stride loop. Persistent blocks keep every SM streaming to the end; one-shot
// blocks ran in waves, and weight tiles in blocks of their own could not share an SM with the
// stages and ran after them. `ch` = channels of x; every block calls it with the same arguments.
constexpr int kRingStages = 3;
constexpr int kRingStageBytes = 16384;
constexpr int kRingBlocksPerSm = 4;  // 3 stages of 16 KB each; <= 64 registers a thread

// The tiles cover the positions [q_lo, q_hi) of every image's volume (q_lo a multiple of the tile
// length); the weight tiles and the remaining items are taken only when `whole` is set. kStages:
// the ring's depth (3; or 1, no copies ahead: the light form that runs beside a GEMM CTA).
template <int kEB, int kCG, int kRotRows, int kRotB, int kStages, class TileFn>
__device__ __forceinline__ void pack_ring(const ConvParams& p, const PackPlan& q, long long x_tiles,
                                          long long q_lo, long long q_hi, bool whole, int ch,
                                          uint8_t* raw, TileFn&& tile_fn) {
  constexpr int kRowB = kRingStageBytes / kCG;  // bytes of a stage row
  constexpr int kTP = kRowB / kEB;              // positions of a tile
  constexpr int kChunks = kRingStageBytes / 16 / 256;  // 16-byte copies per thread per tile
  static_assert(kRowB % 128 == 0 && kRotB % 16 == 0 && kChunks * 256 * 16 == kRingStageBytes,
                "tile");
  static_assert(kRingStageBytes >= kWTileBytes, "a weight tile uses one stage");
  static_assert(kStages == 1 || kStages == 3, "ring depth");
  static_assert(kPackTilePositions % kTP == 0, "range starts fall on tile boundaries");
  const long long b = blockIdx.x, nb = gridDim.x;
  const long long n_tiles = x_tiles + (whole ? q.w_blocks : 0);
  const long long dhw = (long long)p.D * p.H * p.W;
  const long long pt = (q_hi - q_lo + kTP - 1) / kTP;
  const int cgn = ch / kCG;
  auto tile_at = [&](long long t, int& valid, long long& q0, int& n, int& c0) {
    const long long pi = t % pt, rest = t / pt;  // positions fastest, then channel groups, images
    n = (int)(rest / cgn);
    c0 = (int)(rest % cgn) * kCG;
    q0 = q_lo + pi * kTP;
    valid = q_hi - q0 < kTP ? (int)(q_hi - q0) : kTP;  // valid * kEB is a multiple of 16
    return p.x + (((long long)n * ch + c0) * dhw + q0) * kEB;
  };
  auto issue = [&](long long t, uint8_t* stage) {  // cp.async copies of x tile t, no wait
    int valid, n, c0;
    long long q0;
    const uint8_t* src = tile_at(t, valid, q0, n, c0);
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
      const int c16 = threadIdx.x + 256 * i;
      const int r = c16 / (kRowB / 16), s = c16 - r * (kRowB / 16);  // row (channel), chunk
      if (16 * s < valid * kEB)
        cp_async_16_zfill(
            smem_u32(stage + r * kRowB + ((16 * s + (r / kRotRows) * kRotB) & (kRowB - 1))),
            src + (long long)r * dhw * kEB + 16 * s, 16);
    }
  };
  if constexpr (kStages == 3) {
    if (b < x_tiles) issue(b, raw);
    cp_async_commit();
    if (b + nb < x_tiles) issue(b + nb, raw + kRingStageBytes);
    cp_async_commit();
  }
  int sidx = 0;
  for (long long t = b; t < n_tiles; t += nb) {
    uint8_t* stage = raw + sidx * kRingStageBytes;
    if constexpr (kStages == 3) {
      const long long t2 = t + 2 * nb;  // into the stage freed at the end of the last step
      if (t2 < x_tiles) issue(t2, raw + ((sidx + 2) % kRingStages) * kRingStageBytes);
      cp_async_commit();
      cp_async_wait_group<2>();  // this thread's copies of tile t have landed
    } else {
      if (t < x_tiles) issue(t, stage);
      cp_async_commit();
      cp_async_wait_group<0>();
    }
    __syncthreads();  // and everyone else's
    if (t >= x_tiles) {
      pack_w_tile(p, q, t - x_tiles, stage);  // nothing is in flight into this stage
    } else {
      int valid, n, c0;
      long long q0;
      tile_at(t, valid, q0, n, c0);
      tile_fn(static_cast<const uint8_t*>(stage), valid, q0, n, c0);
    }
    __syncthreads();  // the stage is free for the copies kStages tiles on
    sidx = (sidx + 1) % kStages;
  }
  cp_async_wait_all();
  if (!whole) return;
  const PackCtx c = pack_ctx(p, q);
  const long long total = c.e3 + q.w_items;
  for (long long g = c.e1 + b * blockDim.x + threadIdx.x; g < total; g += nb * blockDim.x)
    pack_rest_item(p, q, c, g);
}

// Byte offset in the channels-last copy of position qq of image n's volume, channel byte cb0. The
// ring kernels run only for D*H*W < 2^31, so the position splits into (d, h, w) with 32-bit
// unsigned divisions (a 64-bit division is a long subroutine, and there is one per item).
__device__ __forceinline__ long long xp_offset(const ConvParams& p, int n, long long qq, int cb0) {
  const unsigned u = (unsigned)qq, W = (unsigned)p.W, H = (unsigned)p.H;
  const unsigned dh = u / W, wq = u - dh * W;
  const unsigned dq = dh / H, hq = dh - dq * H;
  return ((((long long)n * p.Dp + dq + p.pk_pd) * p.Hp + hq + p.pk_ph) * p.Wp + wq + p.pk_pw) *
             p.C + cb0;
}

// Tiled transpose of an NCDHW x into the channels-last copy, for e4m3 bytes (kEB = 1) and for the
// BF16 twin's bfloat16 elements (kEB = 2), without rounding anything: the elements move as they
// are. Shapes: W % 4 == 0, D*H*W*kEB % 16 == 0, C % kCG == 0. A tile is 128 (e4m3, C % 128 == 0)
// or 64 channels. Each thread takes one (16-byte channel block, 4-position group) of a tile: one
// 4-position word (e4m3: 4 bytes, bfloat16: 8 bytes) from each of the block's 16 / kEB channel
// rows, through byte permutes into four 16-byte chunks, one per position. The threads of a
// position are adjacent in the warp, so one store instruction writes whole kCG * kEB-byte runs of
// pixel rows. Rows rotate by 128 / (channel blocks of a tile) bytes per channel block, so that
// the words a warp (bfloat16: a half-warp) reads fall in 32 different banks. The item path this
// replaced for these shapes held 16 x 16 bytes a thread in registers (100 registers, two blocks an
// SM): 31.4 us for the large layer's x, against 18.5 us for each further image of the same size.
template <int kEB, int kCG, int kStages>
__global__ void __launch_bounds__(256, kRingBlocksPerSm) pack_x_transpose_kernel(
    ConvParams p, PackPlan q, long long x_tiles, long long q_lo, long long q_hi, int whole) {
  pdl_launch_dependents();  // the implicit GEMM may start its prologue while the pack runs
  constexpr int kRowB = kRingStageBytes / kCG;
  constexpr int kChB = 16 / kEB;   // channels of a 16-byte block
  constexpr int kCB = kCG / kChB;  // channel blocks of a tile
  constexpr int kRotB = 128 / kCB;
  static_assert(kEB == 1 || kEB == 2, "element bytes");
  static_assert(kCB * (kRowB / kEB / 4) == 256, "one (channel block, position group) per thread");
  extern __shared__ __align__(16) uint8_t raw[];  // [kRingStages][kCG][kRowB] bytes
  const int cb = threadIdx.x % kCB;  // this thread's channel block and position group
  const int qg = threadIdx.x / kCB;
  pack_ring<kEB, kCG, kChB, kRotB, kStages>(p, q, x_tiles, q_lo, q_hi, whole != 0, p.C / kEB,
                                             raw,
      [&](const uint8_t* stage, int valid, long long q0, int n, int c0) {
    if (4 * qg >= valid) return;
    // the group's word in each of its rows, at the rotated byte column
    const uint8_t* rows = stage + (kChB * cb) * kRowB + ((4 * kEB * qg + cb * kRotB) & (kRowB - 1));
    uint32_t o[4][4];  // o[position][word of the 16-byte chunk]
    if constexpr (kEB == 1) {
      uint32_t v[16];  // v[m]: positions 4qg..4qg+3 of channel 16cb + m
#pragma unroll
      for (int m = 0; m < 16; ++m) v[m] = *reinterpret_cast<const uint32_t*>(rows + m * kRowB);
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        uint32_t tt[4];
        transpose4x4(v + 4 * bb, tt);
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j][bb] = tt[j];
      }
    } else {
      uint2 v[8];  // v[m]: positions 4qg, 4qg+1 (.x) and 4qg+2, 4qg+3 (.y) of channel 8cb + m
#pragma unroll
      for (int m = 0; m < 8; ++m) v[m] = *reinterpret_cast<const uint2*>(rows + m * kRowB);
#pragma unroll
      for (int mm = 0; mm < 4; ++mm) {  // channel pair (2mm, 2mm + 1)
        o[0][mm] = __byte_perm(v[2 * mm].x, v[2 * mm + 1].x, 0x5410);
        o[1][mm] = __byte_perm(v[2 * mm].x, v[2 * mm + 1].x, 0x7632);
        o[2][mm] = __byte_perm(v[2 * mm].y, v[2 * mm + 1].y, 0x5410);
        o[3][mm] = __byte_perm(v[2 * mm].y, v[2 * mm + 1].y, 0x7632);
      }
    }
    // W % 4 == 0 keeps the group's four positions in one row
    uint8_t* dst = p.xp + xp_offset(p, n, q0 + 4 * qg, c0 * kEB + 16 * cb);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4*>(dst + (long long)j * p.C) =
          make_uint4(o[j][0], o[j][1], o[j][2], o[j][3]);
  });
}

bool pack_transposes_x(const ConvParams& p) {
  const long long dhw = (long long)p.D * p.H * p.W;
  return p.xp != nullptr && !p.x_cl && p.x_src_type == kSrcE4m3 && p.W % 4 == 0 &&
         (dhw * p.elem_bytes) % 16 == 0 && (p.C / p.elem_bytes) % 64 == 0 && dhw < (1LL << 31);
}

// The light form (kStages == 1) is launched as a programmatic dependent of the GEMM before it: it
// starts once every CTA of that GEMM has triggered its dependents, and never waits for it.
template <int kEB, int kCG, int kStages>
static cudaError_t launch_transpose(const ConvParams& p, const PackPlan& q, long long x_tiles,
                                    long long blocks, long long q_lo, long long q_hi, bool whole,
                                    cudaStream_t stream) {
  auto kernel = pack_x_transpose_kernel<kEB, kCG, kStages>;
  // one tile per block: only the first stage is used
  const long long n_tiles = x_tiles + (whole ? q.w_blocks : 0);
  const size_t smem = (size_t)kRingStageBytes * (blocks < n_tiles ? kStages : 1);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = kStages == 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p, q, x_tiles, q_lo, q_hi, whole ? 1 : 0);
}

cudaError_t launch_pack_range(const ConvParams& p, long long q_lo, long long q_hi, bool whole,
                              bool light, cudaStream_t stream) {
  const PackPlan q = pack_plan(p);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int ch = p.C / p.elem_bytes;  // channels
  const int cg = p.elem_bytes == 1 && ch % 128 == 0 ? 128 : 64;
  const long long tp = kRingStageBytes / cg / p.elem_bytes;
  const long long x_tiles = q_hi > q_lo ? (long long)p.N * (ch / cg) * ((q_hi - q_lo + tp - 1) / tp)
                                        : 0;
  const long long n_tiles = x_tiles + (whole ? q.w_blocks : 0);
  if (n_tiles == 0 && !whole) return cudaSuccess;
  long long blocks = std::min<long long>(n_tiles, (long long)sms * (light ? 1 : kRingBlocksPerSm));
  if (blocks < 1) blocks = 1;
  if (light) {
    if (p.elem_bytes == 2)
      return launch_transpose<2, 64, 1>(p, q, x_tiles, blocks, q_lo, q_hi, whole, stream);
    return cg == 128 ? launch_transpose<1, 128, 1>(p, q, x_tiles, blocks, q_lo, q_hi, whole, stream)
                     : launch_transpose<1, 64, 1>(p, q, x_tiles, blocks, q_lo, q_hi, whole, stream);
  }
  if (p.elem_bytes == 2)
    return launch_transpose<2, 64, 3>(p, q, x_tiles, blocks, q_lo, q_hi, whole, stream);
  return cg == 128 ? launch_transpose<1, 128, 3>(p, q, x_tiles, blocks, q_lo, q_hi, whole, stream)
                   : launch_transpose<1, 64, 3>(p, q, x_tiles, blocks, q_lo, q_hi, whole, stream);
}

// Direct route: the explicit A = im2col(x), [npq][kg] bytes with K_gemm in the caller's KCTRS
// order: A[row][e] = x[n, c, od*sd + t - pd, oh*sh + r - ph, ow*sw + s - pw] for element
// e = c*taps + tap, zero where the tap falls outside the volume. The weights are not touched: the
// implicit GEMM reads them as they are. A thread writes one 16-byte chunk of a row; consecutive
// threads take consecutive rows of the same chunk, so the (c, t, r, s) walk of a warp is uniform
// and each of its loads reads 32 neighbouring output positions' taps. kType: kSrcE4m3 copies the
// elements (e4m3 bytes, or the BF16 twin's bfloat16 halves); kSrcF32 / kSrcBf16 quantise fp32 /
// bfloat16 values with the device scale *scale_x. kEl: bytes of an output element.
template <int kType, int kEl>
__global__ void __launch_bounds__(256) im2col_kernel(ConvParams p) {
  pdl_launch_dependents();  // the implicit GEMM may start its prologue while this runs
  constexpr bool kQuant = kType != kSrcE4m3;
  constexpr int el = kEl;
  constexpr int per = 16 / el;  // elements per 16-byte chunk
  const int cpr = p.kg / 16;                 // chunks per row
  const long long total = (long long)p.npq * cpr;
  const int taps = p.taps, RS = p.R * p.S, HW = p.H * p.W, DHW = p.D * HW;
  const int c_el = p.C / el;  // channels
  const float qs = kQuant ? __ldg(p.scale_x) : 1.0f;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(g % p.npq);
    const int q = (int)(g / p.npq);
    const int n = row / p.dhw;
    const int pix = row - n * p.dhw;
    const int ow = pix % p.Wo;
    const int t2 = pix / p.Wo;
    const int oh = t2 % p.Ho;
    const int od = t2 / p.Ho;
    const int d0 = od * p.sd - p.pd, h0 = oh * p.sh - p.ph, w0 = ow * p.sw - p.pw;
    const long long img = (long long)n * c_el * DHW;  // x index of x[n, 0, 0, 0, 0]
    const int e0 = q * per;
    int c = e0 / taps, tap = e0 - c * taps;
    int t = tap / RS;
    const int rs = tap - t * RS;
    int r = rs / p.S, s = rs - r * p.S;
    uint32_t v[4] = {0u, 0u, 0u, 0u};
    float f[per];
#pragma unroll
    for (int j = 0; j < per; ++j) {
      const bool in = (unsigned)(d0 + t) < (unsigned)p.D && (unsigned)(h0 + r) < (unsigned)p.H &&
                      (unsigned)(w0 + s) < (unsigned)p.W;
      const long long idx = img + (long long)c * DHW + ((d0 + t) * p.H + (h0 + r)) * p.W + (w0 + s);
      if (kQuant) {
        f[j] = in ? src_value(p.x, kType, idx) : 0.0f;
      } else if (in) {
        const uint32_t e = el == 1 ? (uint32_t)__ldg(p.x + idx)
                                   : (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(p.x) + idx);
        v[(j * el) >> 2] |= e << (((j * el) & 3) * 8);
      }
      if (++tap == taps) {
        tap = t = r = s = 0;
        ++c;
      } else if (++s == p.S) {
        s = 0;
        if (++r == p.R) {
          r = 0;
          ++t;
        }
      }
    }
    if constexpr (kQuant) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        v[k] = quant4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3], qs);
    }
    *reinterpret_cast<uint4*>(p.xp + (long long)row * p.kg + (long long)q * 16) =
        make_uint4(v[0], v[1], v[2], v[3]);
  }
}

cudaError_t launch_pack(const ConvParams& p, cudaStream_t stream) {
  if (p.route == kRouteDirect) {  // the explicit im2col of x; the weights stay as they are
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long total = (long long)p.npq * (p.kg / 16);
    long long blocks = (total + 255) / 256;
    if (blocks > (long long)sms * 16) blocks = (long long)sms * 16;
    if (blocks < 1) blocks = 1;
    if (p.x_src_type == kSrcF32)
      im2col_kernel<kSrcF32, 1><<<(unsigned)blocks, 256, 0, stream>>>(p);
    else if (p.x_src_type == kSrcBf16)
      im2col_kernel<kSrcBf16, 1><<<(unsigned)blocks, 256, 0, stream>>>(p);
    else if (p.elem_bytes == 2)
      im2col_kernel<kSrcE4m3, 2><<<(unsigned)blocks, 256, 0, stream>>>(p);
    else
      im2col_kernel<kSrcE4m3, 1><<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
  }
  const PackPlan q = pack_plan(p);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long cap = (long long)sms * 16;
  const long long rest_items = q.halo_row_items + q.halo_side_items + q.w_items;
  const long long dhw = (long long)p.D * p.H * p.W;
  if (q.x_items > 0 && !q.copy && p.elem_bytes == 1 && p.x_src_type != kSrcE4m3) {
    // an NCDHW x quantised on the way: the tiled transpose, plus blocks for the remaining items
    // and the weight tiles. bfloat16 x: persistent blocks over 32-channel tiles in two 32 KB
    // stages (large layer step 332 -> 323 us against one tile per block); fp32 x: one 32-channel
    // tile (48 KB) per block (two-stage forms of 512-position tiles measured 364 us with 16
    // channels, 399 us with 32 on one block per SM, against 362 us for one 64 KB tile per block;
    // 384-position tiles, 4 blocks an SM, then took the pack from 73.9 to 69.8 us). The ring of
    // the plain transposes (16 KB tiles of
    // 32 channels x 128 / 256 positions, 4 blocks an SM, one 16-channel column of a position a
    // thread, a position's 32 bytes written by one instruction) measured slower here, bit-exact
    // all the same: the large layer's pack 74.5 -> 82.3 us from fp32, 61.7 -> 67.7 us from
    // bfloat16.
    const bool f32 = p.x_src_type == kSrcF32;
    const int ct = p.C % 32 == 0 ? 32 : 16;
    const long long tp = f32 ? tile_positions<kSrcF32>() : tile_positions<kSrcBf16>();
    const long long x_tiles = (long long)p.N * (p.C / ct) * ((dhw + tp - 1) / tp);
    const long long tile_blocks =
        f32 ? x_tiles
            : std::min<long long>(x_tiles, (long long)sms * tiled_blocks_per_sm<kSrcBf16>());
    long long rest_blocks = (rest_items + 255) / 256;
    if (rest_blocks > cap) rest_blocks = cap;
    if (f32 && ct == 32)
      return launch_tiled_ct<kSrcF32, 32>(p, q, x_tiles, tile_blocks, rest_blocks, stream);
    if (f32) return launch_tiled_ct<kSrcF32, 16>(p, q, x_tiles, tile_blocks, rest_blocks, stream);
    if (ct == 32)
      return launch_tiled_ct<kSrcBf16, 32>(p, q, x_tiles, tile_blocks, rest_blocks, stream);
    return launch_tiled_ct<kSrcBf16, 16>(p, q, x_tiles, tile_blocks, rest_blocks, stream);
  }
  if (q.x_items > 0 && pack_transposes_x(p)) {
    // e4m3 bytes or the twin's bfloat16, NCDHW: the tiled transpose; the same blocks take the
    // weight tiles and the remaining items
    return launch_pack_range(p, 0, dhw, true, false, stream);
  }
  const long long total = q.x_items + rest_items;
  long long item_blocks = (total + 255) / 256;
  if (item_blocks > cap) item_blocks = cap;
  if (item_blocks + q.w_blocks < 1) item_blocks = 1;
  pack_kernel<<<(unsigned)(item_blocks + q.w_blocks), 256,
                q.w_blocks > 0 ? (size_t)kWTileBytes : 0, stream>>>(p, q, (int)item_blocks);
  return cudaGetLastError();
}

// Split-K reduction of the split tiles (full_tiles..m_tiles*n_tiles-1):
// y = bf16(scale * sum_{split = 0..splits-1} partial[split]) in ascending split order, so the
// result is bitwise reproducible for a fixed plan. One thread per (tile, column, row); the stores
// carry the same guards as the main epilogue (real output row, col < K).
template <bool kRowChk>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(ConvParams p) {
  const long long per_tile = (long long)p.block_n * p.block_m;
  const long long total = ((long long)p.m_tiles * p.n_tiles - p.full_tiles) * per_tile;
  pdl_wait_primary();  // the partials of the implicit GEMM, complete and visible
  const float scale = __ldg(p.scale_x) * __ldg(p.scale_w);
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(g % p.block_m);
    const int col_l = (int)((g / p.block_m) % p.block_n);
    const long long t = g / per_tile;  // index among the split tiles
    const long long tile = p.full_tiles + t;
    const int n_tile = (int)(tile % p.n_tiles);
    const int m_tile = (int)(tile / p.n_tiles);
    const int col = n_tile * p.block_n + col_l;
    if (col >= p.K) continue;
    const RowDest dst = row_dest(p, m_tile, row);
    if (kRowChk && !dst.valid) continue;
    const float* src = p.partials + ((t * p.splits) * p.block_n + col_l) * p.block_m + row;
    // eight loads in flight at a time; the additions stay in ascending split order
    float acc = 0.0f;
    int s = 0;
    for (; s + 8 <= p.splits; s += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __ldcg(src + (long long)(s + j) * per_tile);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc += v[j];
    }
    for (; s < p.splits; ++s) acc += __ldcg(src + (long long)s * per_tile);
    const __nv_bfloat16 b = __float2bfloat16_rn(acc * scale);
    p.y[dst.y_off + (long long)col * p.dhw] = *reinterpret_cast<const uint16_t*>(&b);
    count_write(p, dst.y_off + (long long)col * p.dhw);
  }
}

cudaError_t launch_splitk_reduce(const ConvParams& p, bool row_chk, cudaStream_t stream) {
  const long long total =
      ((long long)p.m_tiles * p.n_tiles - p.full_tiles) * p.block_n * p.block_m;
  if (total <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)sms * 16;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return row_chk ? cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<true>, p)
                 : cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<false>, p);
}

}  // namespace c3d
