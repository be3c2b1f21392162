// Shared constants, layouts and numeric helpers of the CUDA path.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------- geometry
constexpr int kTopK = MOE_TOPK;
constexpr int kUnitRows = MOE_UNIT_ROWS;   // MMA N: pair rows per unit
constexpr int kTileM = 128;                // MMA M: weight rows per tile
constexpr int kChunkK = 128;               // K elements per weight stage
constexpr int kBlock = 32;                 // MX block (one E8M0 scale)
constexpr int kTileBytes = kTileM * kChunkK / 2;      // 8192: packed e2m1
constexpr int kStageWeightBytes = 2 * kTileBytes;     // two tiles per stage
constexpr int kScaleAtomBytes = 512;       // 32 rows x 16 B (128 rows x 4 k-blocks)
constexpr int kStageBytes = kStageWeightBytes + 2 * kScaleAtomBytes;  // 17408
constexpr int kStageSmemWeights = 2 * kTileM * kChunkK;  // 32768: e2m1 in 8-bit slots
constexpr int kActImageBytes = kUnitRows * kChunkK;      // 1024: one 128B-swizzle atom
constexpr int kHiddenChunkBytes = kActImageBytes + kScaleAtomBytes;  // codes + scale atom

constexpr int kRingStages = 6;
constexpr int kMmaWarps = 4;              // MMA issuers: (tile 0/1) x (K-steps 0-1 / 2-3)
constexpr int kAccSets = 4;               // TMEM accumulator sets
constexpr int kAccSetColumns = kMmaWarps * 8;       // one N = 8 accumulator per issuer
constexpr int kTmemScaleBase = kAccSets * kAccSetColumns;  // 128: per-slot scale columns
constexpr int kSlotScaleColumns = kMmaWarps * 8;    // per issuer: A atom (4) + B atom (4)
// FC2 hidden-vector scale atoms, copied once per unit: per issuer, 2 image
// buffers x kMaxInterChunks chunks x 4 columns, after the per-slot columns.
constexpr int kTmemHiddenScaleBase = kTmemScaleBase + kRingStages * kSlotScaleColumns;  // 320
constexpr int kHiddenScaleColumns = 2 * 4 * 4;  // per issuer
constexpr int kTmemColumns = 512;
static_assert(kTmemHiddenScaleBase + kMmaWarps * kHiddenScaleColumns <= kTmemColumns,
              "TMEM columns: accumulators, slot scales and hidden scales fit");
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp0 = 1;              // warps 1..4
constexpr int kGatherWarp = 5;
constexpr int kEpilogueWarp0 = 6;         // warps 6..9: the epilogue warpgroup
constexpr int kThreads = 320;             // 10 warps
// The grid kernel adds two scale-copy warps (10, 11): they copy each stage's
// three scale atoms (weights of tile 0 and 1, activations) into TMEM once
// for all four issuers, which then issue only MMAs and a commit per stage.
constexpr int kCopierWarp0 = 10;
constexpr int kCopiers = 2;
constexpr int kGridThreads = 384;         // 12 warps
constexpr int kMaxInterChunks = MOE_MAX_INTER / kChunkK;  // 4
constexpr int kMaxGrid = 256;             // partition table capacity (CTAs)
constexpr int kMaxSpanCtas = 512;         // launch-clock slots: CTAs of any experts launch

// The grid kernel's units: the table's 8-row units for calls of at most 8
// tokens, else pairs of them. An N = 16 MMA costs its issuing thread as much
// as an N = 8 one, so a 16-row unit streams an expert's weights once for up
// to 16 of its tokens. A pair-table entry: bits 0-19 the first unit, 20-29
// the expert, bit 31 set when the next unit is the same expert's (rows 8-15).
constexpr uint32_t kWideFirstMask = 0xFFFFFu;
__host__ __device__ constexpr uint32_t wide_entry(int first, int expert, bool paired) {
  return static_cast<uint32_t>(first) | (static_cast<uint32_t>(expert) << 20) | (paired ? 1u << 31 : 0u);
}
static_assert(MOE_MAX_EXPERTS <= 1024, "the pair-table entry holds a 10-bit expert");

// Per-unit-size constants of the grid kernel: 16-row units take a 5-slot ring
// (the images and staging double; a 5-slot ring streams as fast at 152 CTAs)
// and 3 accumulator sets of 4 x 16 TMEM columns.
template <int R>
struct Rows {
  static constexpr int kSlots = R == 8 ? kRingStages : 5;
  static constexpr int kSets = R == 8 ? kAccSets : 3;
  static constexpr int kImage = R * kChunkK;            // activation / hidden image of a K chunk
  static constexpr int kSetColumns = kMmaWarps * R;     // one N = R accumulator per issuer
  static constexpr int kScaleBase = kSets * kSetColumns;
  static constexpr int kHiddenScaleBase = kScaleBase + kSlots * kSlotScaleColumns;
  static_assert(kHiddenScaleBase + kMmaWarps * kHiddenScaleColumns <= kTmemColumns, "TMEM columns");
};

// Byte offset of the 16-byte chunk `c16` (0..7) of row `r` in a 128-byte-
// swizzled image of 8-row, 1024-byte atoms (rows 8-15 are the second atom).
__host__ __device__ constexpr uint32_t swizzle128(uint32_t r, uint32_t c16) {
  return r * 128u + ((c16 ^ (r & 7u)) << 4);
}

// Byte offset of (row r, k-block kb) in a 512-byte scale atom that the
// tensor core's 32x128b scale copy expects: 128 rows x 4 k-blocks.
__host__ __device__ constexpr uint32_t scale_atom(uint32_t r, uint32_t kb) {
  return (r & 31u) * 16u + (r >> 5) * 4u + kb;
}

// Per-layer geometry, shared by host and device.
struct Geometry {
  int E, H, I;
  int KC1;   // FC1 K chunks (H / 128)
  int P1;    // FC1 tile pairs: 128 gate rows + the matching 128 up rows (ceil(I / 128))
  int NQ;    // FC2 jobs per unit: tile pairs of 256 output rows (H / 256)
  int KC2;   // FC2 K chunks (ceil(I / 128))
  int SPE;   // stages per expert: P1 * KC1 + NQ * KC2
  int hidden_bytes;  // per-unit hidden image: KC2 * (1024 codes + 512 scales)
  int floor_rule;    // hidden requant: floor(log2 amax) - 8 iff 2I == 768
};

inline Geometry make_geometry(int E, int H, int I) {
  Geometry g;
  g.E = E;
  g.H = H;
  g.I = I;
  g.KC1 = H / kChunkK;
  g.P1 = (I + kTileM - 1) / kTileM;
  g.NQ = H / (2 * kTileM);
  g.KC2 = (I + kChunkK - 1) / kChunkK;
  g.SPE = g.P1 * g.KC1 + g.NQ * g.KC2;
  g.hidden_bytes = g.KC2 * kHiddenChunkBytes;
  g.floor_rule = (2 * I == 768) ? 1 : 0;
  return g;
}

// Unit-table capacity for a batch: sum_e ceil(n_e / 8) <= 2B + min(E, 16B).
inline int unit_capacity(int batch, int experts) {
  int pairs = batch * kTopK;
  return 2 * batch + (experts < pairs ? experts : pairs);
}

// ------------------------------------------------------------- numerics
// 2^e as an exact float for e in [-149, 127].
__device__ __forceinline__ float pow2f(int e) {
  if (e >= -126) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  return __uint_as_float(1u << (e + 149));
}

// Shared exponent of an MXFP8 block from its largest magnitude (an FP32
// value): ceil rule = smallest E with amax <= 448 * 2^E, floor rule =
// floor(log2 amax) - 8; zero (or FP32-subnormal) amax gives -127; clamped
// to [-127, 127]. 448 = 1.75 * 2^8, so with amax = m * 2^q (1 <= m < 2) the
// ceil rule is q - 8, plus one when m > 1.75 (mantissa bits above 0x600000).
__device__ __forceinline__ int mx_exponent(float amax, bool floor_rule) {
  uint32_t bits = __float_as_uint(amax) & 0x7FFFFFFFu;
  int biased = static_cast<int>(bits >> 23);
  if (biased == 0) return -127;
  int E = biased - 127 - 8;
  if (!floor_rule && (bits & 0x7FFFFFu) > 0x600000u) E += 1;
  return E < -127 ? -127 : (E > 127 ? 127 : E);
}

// e4m3 code of v: round to nearest even, saturate to +-448, keep the sign.
__device__ __forceinline__ uint8_t e4m3_code(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// Device status word: the first error code wins.
__device__ __forceinline__ void report(int32_t* status, int code) {
  atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

}  // namespace moe
