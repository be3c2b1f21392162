// Kernel argument blocks and host launchers shared by the translation units.
#pragma once

#include "common.cuh"

namespace moe {

// Prep kernel: MXFP8 activation plan (blocks 0 .. quant_blocks-1) and the
// unit table (the last block), as requested by `roles`.
enum PrepRoles : int { kPrepQuantize = 1, kPrepGroup = 2 };

struct PrepArgs {
  const uint16_t* x;        // BF16 [B, H]
  const int32_t* ids;       // [B, 16]
  int B, H, E, P1, KC2, unit_cap;
  uint8_t* plan_codes;      // [B, H]
  uint8_t* plan_scales;     // [B, H / 32]
  int32_t* unit_count;      // [1]
  int32_t* unit_expert;     // [unit_cap]
  int16_t* unit_rows;       // [unit_cap, 8]
  uint32_t* wide_units;     // [unit_cap]: the pairs of units (see kWideFirstMask)
  uint32_t* item_counters;  // [unit_cap * P1], cleared per call
  uint32_t* hidden_flags;   // [unit_cap * KC2], cleared per call
  uint8_t* pair_kept;       // [B * 16] or null: 1 where the pair got a unit row
  int32_t* status;
  int roles;
  int quant_blocks;
  // Early start (the previous launch on the stream was another handle's
  // call): the blocks write without waiting for the previous grid, the last
  // one raises *ready to seq (release), and every block then waits for the
  // previous grid before it ends.
  int early;
  uint32_t seq;
  uint32_t* ready;            // [1]: the number of the last call whose tables are out
  uint32_t* arrive;           // [1]: blocks done writing (zero at rest)
  // Its own experts kernel follows at once (moe_run): let it launch at this
  // grid's start. Otherwise (moe_quantize, moe_group) the next launch waits
  // for this grid's end.
  int chained;
};

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t stream);
int prep_quant_blocks(int batch, int hidden);
int prep_group_smem_bytes(int experts);

// Persistent experts kernel.
struct ExpertsArgs {
  CUtensorMap wmap;           // 3-D map over the stage blocks (first: 64-byte aligned)
  const uint8_t* stages;      // [E * SPE] blocks of kStageBytes
  const int32_t* ids;         // [B, 16] routing ids of the call, or null: lets the cluster
                              // variant's producer find its unit without the prep grid
  uint8_t* plan_codes;        // [B, H] (the small-batch kernel writes it, the others read it)
  uint8_t* plan_scales;       // [B, H / 32]
  int32_t* unit_count;         // [0] units, [1] pairs of units
  int32_t* unit_expert;
  int16_t* unit_rows;
  const uint32_t* wide_units;  // [unit_cap]: the 16-row units of calls of more than 8 tokens
  uint32_t* item_counters;
  uint32_t* hidden_flags;
  float* partials;            // [grid, 2 halves, 2 tiles, R rows, 128 weight rows]
  uint8_t* hidden;            // [unit_cap, hidden_bytes]
  uint16_t* out;              // BF16 [B * 16, H]
  int32_t* status;
  int B;                      // tokens of the call
  Geometry g;
  uint64_t timeout_ns;
  int withhold_unit;          // test hook: never publish this unit's hidden (-1 = off)
  int withhold_image;         // test hook (grid kernel): never deliver this unit's hidden
                              // image to shared memory (-1 = off)
  uint64_t* span;             // or null: launch clock, [CTA][start, end] (moe_debug_kernel_span)
  // Small-batch kernel only (the call is that one launch):
  const uint16_t* x;          // BF16 [B, H]: quantized to MXFP8 in the kernel
  uint32_t* piece_sums;       // [2 parities][seg_cap][kSmallPieceWords]: FC1 segment sums, sentinel at rest
  uint32_t* piece_readers;    // [2][seg_cap]: consumers that read the segment, zero at rest
  uint32_t* small_counters;   // [2 parities][4]: [0] segments claimed (zero at rest)
  uint8_t* pair_kept;         // [B * 16] or null: 1 where the pair got a unit row
  uint64_t* trace;            // or null: per-CTA phase stamps (builds with MOE_TRACE only)
  // Grid kernel, early start: read the tables once *ready == seq instead of
  // waiting for the prep grid to end; wait for it only before the first
  // output row (its end implies the previous experts grid's). The last CTA
  // to see the flag puts it back to 0, so that a replay of the same call (a
  // CUDA graph keeps seq) waits for its own prep grid.
  int early;
  uint32_t seq;
  uint32_t* ready;
  uint32_t* passed;           // [1]: CTAs that saw the flag (zero at rest)
  int skew;                   // FC1 ranges skewed toward the low CTAs (see Split)
  int seg_cap;                // segment slots per parity
  int piece_words;            // words per segment slot (2 x the batch bound x 128)
  int parity;                 // which half of the slots and counters this call uses
};

int experts_smem_bytes(const Geometry& g, int unit_rows = 8);
// The most dynamic shared memory any experts kernel takes for this layer.
int experts_max_smem_bytes(const Geometry& g);
bool experts_layout_aligned(const Geometry& g);
cudaError_t experts_configure(const Geometry& g);
cudaError_t experts_occupancy(const Geometry& g, int* blocks_per_sm);
// Work split of the cluster variant, computed on the host per launch: CTA r
// of a cluster runs FC1 stages [fc1[r], fc1[r + 1]) and FC2 jobs
// [fc2[r], fc2[r + 1]) of its unit; FC1 item p is owned by CTA owner[p],
// which receives pieces[p] partial sums, CTA r's into slot[p][r] (-1: none).
struct ClusterPlan {
  int C;
  int fc1[9], fc2[9];
  int owner[kMaxInterChunks], pieces[kMaxInterChunks];
  int8_t slot[kMaxInterChunks][8];
};

// Which experts kernel serves a call: kPathGrid always the persistent grid
// kernel; kPathSmall (default) the small-batch kernel for calls of one or two
// tokens whose routing ids are given and whose split fits it (small_fits),
// else the grid kernel; kPathCluster the cluster variant for one or two
// tokens where the shape fits it, else the grid kernel; kPathSmallWide the
// small-batch kernel for calls of up to kSmallMaxBatch tokens where it fits.
enum ExpertsPath : int { kPathGrid = 0, kPathSmall = 1, kPathCluster = 2, kPathSmallWide = 3 };
cudaError_t launch_experts(const ExpertsArgs& a, int grid, cudaStream_t stream, bool pdl,
                           int path, bool small);
int cluster_size_for(const Geometry& g, int batch);  // 0: the grid kernel serves this call
bool small_fits(const Geometry& g, int batch, int grid);
// The small-batch kernel's build for a call: kSmallPacked (one or two tokens,
// x and hidden images 256 bytes apart, 3-slot ring), kSmallWide (up to 8
// tokens, 2-slot ring) or 0 when neither fits the layer.
constexpr int kSmallPacked = 1, kSmallWide = 2;
int small_build(const Geometry& g, int batch, int grid);
cudaError_t small_configure();
cudaError_t launch_small(const ExpertsArgs& a, int grid, cudaStream_t stream, bool pdl);
constexpr int kSmallMaxBatch = 8;  // calls of up to 8 tokens may take the small-batch kernel
// Whether a handle's path value sends a call of `batch` tokens to the
// small-batch kernel (where small_fits also holds).
inline bool small_path_serves(int path, int batch) {
  return (path == kPathSmall && batch <= 2) || (path == kPathSmallWide && batch <= kSmallMaxBatch);
}
// The small-batch kernel's FC1 segment slots: gate and up FP32 sums of up to
// kSmallMaxBatch token rows per 128-row tile (one segment: an even share of the
// K chunks of one item, about kSegChunks of them), and a read count per slot,
// in two halves that consecutive calls alternate. A slot holds kPieceSentinel
// in every word between uses (no finite or canonical-NaN FP32 sum has this
// pattern), so a consumer polls the sums themselves.
constexpr int kSmallPieceWords = 2 * kSmallMaxBatch * 128;
constexpr uint32_t kPieceSentinel = 0xFFFFFFFFu;
constexpr int kSegChunks = 10;
// Segments per item: KC1 / kSegChunks rounded, at least one; segment s of an
// item covers K chunks [s * KC1 / spi, (s + 1) * KC1 / spi).
__host__ __device__ inline int small_spi(int kc1) {
  const int n = (2 * kc1 + kSegChunks) / (2 * kSegChunks);
  return n > 1 ? n : 1;
}
// Segment slots per parity of a layer: 128 units of ceil(I / 128) items.
inline int small_seg_cap(const Geometry& g) { return kSmallMaxBatch * kTopK * g.P1 * small_spi(g.KC1); }
inline size_t small_piece_bytes(const Geometry& g) { return 2 * static_cast<size_t>(small_seg_cap(g)) * kSmallPieceWords * 4; }
inline size_t small_reader_bytes(const Geometry& g) { return 2 * static_cast<size_t>(small_seg_cap(g)) * 4; }
constexpr size_t kSmallCounterBytes = 2 * 4 * 4;

// Routing-weighted combine of each token's 16 rows (after the experts kernel).
struct CombineArgs {
  const uint16_t* rows;     // BF16 [B * 16, H]: the per-pair rows of the run
  const float* weights;     // [B, 16]
  const uint8_t* kept;      // [B * 16]: 1 where the pair's row was written
  uint16_t* out;            // BF16 [B, H]
  int B, H;
};

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream);

// Weight repack into stage blocks.
cudaError_t launch_repack(const uint8_t* w13, const uint8_t* s13, const uint8_t* w2,
                          const uint8_t* s2, const Geometry& g, uint8_t* stages,
                          cudaStream_t stream);

}  // namespace moe
