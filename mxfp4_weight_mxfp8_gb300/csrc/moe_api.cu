// The C ABI (include/moe.h): handle, weight repack, buffers, launches.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "kernels.h"

using moe::Geometry;

struct moe_ctx {
  int device = 0;
  Geometry g{};
  int sms = 0, grid = 0, smem_bytes = 0, unit_cap = 0;
  uint8_t* stages = nullptr;
  size_t stage_bytes = 0;
  uint8_t* workspace = nullptr;
  size_t workspace_bytes = 0;
  uint8_t* plan_codes = nullptr;
  uint8_t* plan_scales = nullptr;
  int32_t* unit_count = nullptr;
  int32_t* unit_expert = nullptr;
  int16_t* unit_rows = nullptr;
  uint32_t* wide_units = nullptr;  // pairs of units: the grid kernel's units above 8 tokens
  uint32_t* item_counters = nullptr;
  uint32_t* hidden_flags = nullptr;
  float* partials = nullptr;
  uint8_t* hidden = nullptr;
  int32_t* status = nullptr;
  int32_t* status_host = nullptr;  // pinned host word: the status read-back stays asynchronous
  int32_t* status_dev = nullptr;   // the word the kernels report into: status, or status_host
  int host_atomics = 0;            // the GPU's atomics on host memory are native (coherent link)
  uint8_t* pair_kept = nullptr;  // [MOE_MAX_BATCH * 16]
  uint16_t* staged = nullptr;    // BF16 [MOE_MAX_BATCH * 16, H]: moe_run_combined's per-pair rows
  uint8_t* io = nullptr;  // device buffers of moe_run_host (x, ids, out), made on first use
  CUtensorMap wmap{};
  uint64_t timeout_ns = 2000000000ull;
  int withhold = -1;
  int withhold_image = -1;
  int path = moe::kPathSmall;  // which experts kernel one- and two-token calls run on
  int small_ok[moe::kSmallMaxBatch + 1] = {};  // [batch]: the small-batch kernel's split fits this layer
  uint64_t* span = nullptr;  // launch clock of the experts kernel: [CTA][start, end]
  uint32_t* piece_sums = nullptr;      // small-batch kernel: FC1 segment slots (sentinel at rest)
  uint32_t* piece_readers = nullptr;   // small-batch kernel: read counts per slot (zero at rest)
  uint32_t* small_counters = nullptr;  // small-batch kernel: segment claims, CTAs done (zero at rest)
  int small_parity = 0;                // the half of the slots and counters the next call takes
  uint32_t* ready = nullptr;   // [0] the number of the last early call whose prep grid wrote its tables
  uint32_t* arrive = nullptr;  // [0] that prep grid's blocks done writing (zero at rest)
  uint32_t* passed = nullptr;  // [0] its experts kernel's CTAs that saw the flag (zero at rest)
  uint32_t seq = 0;            // early calls made
  int span_on = 0;
  uint64_t* trace = nullptr;  // phase stamps (MOE_TRACE builds only)
  int plan_batch = 0, group_batch = 0, grouped = 0, ran = 0;
  uint64_t settings = 0;  // bumped by every setter that changes kernel arguments
  // moe_run_host in place: the call's two launches, captured once per set of
  // host buffers, batch and settings, and replayed as one graph launch.
  cudaStream_t capture_stream = nullptr;
  cudaGraphExec_t host_exec = nullptr;
  const void* host_x = nullptr;
  const void* host_ids = nullptr;
  const void* host_out = nullptr;
  int host_batch = 0;
  uint64_t host_settings = 0;
};

namespace {

thread_local char g_detail[256] = "";

int cuda_fail(cudaError_t e, const char* what) {
  std::snprintf(g_detail, sizeof g_detail, "%s: %s", what, cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

#define MOE_CUDA(call)                                  \
  do {                                                  \
    cudaError_t moe_e_ = (call);                        \
    if (moe_e_ != cudaSuccess) return cuda_fail(moe_e_, #call); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

bool is_device_pointer(const void* p) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged;
}

int encode_weight_map(moe_ctx* h) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  cudaDriverEntryPointQueryResult found{};
  MOE_CUDA(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled",
                                            reinterpret_cast<void**>(&encode), 12000,
                                            cudaEnableDefault, &found));
  if (encode == nullptr || found != cudaDriverEntryPointSuccess) {
    std::snprintf(g_detail, sizeof g_detail, "cuTensorMapEncodeTiled unavailable");
    return MOE_ERR_UNSUPPORTED;
  }
  // Dimension 0: 128 e2m1 values of one row (64 bytes, expanded to 128 in
  // shared memory); dimension 1: the 256 rows of a stage's two tiles;
  // dimension 2: stage blocks. One box = one whole stage.
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(moe::kChunkK), 2u * moe::kTileM,
                              static_cast<cuuint64_t>(h->g.E) * h->g.SPE};
  const cuuint64_t strides[2] = {moe::kChunkK / 2, static_cast<cuuint64_t>(moe::kStageBytes)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(moe::kChunkK), 2u * moe::kTileM, 1u};
  const cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = encode(&h->wmap, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, h->stages, dims, strides,
                      box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_detail, sizeof g_detail, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

void release(moe_ctx* h) {
  if (h == nullptr) return;
  int current = 0;
  cudaGetDevice(&current);
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  cudaFree(h->stages);
  cudaFree(h->workspace);
  cudaFree(h->io);
  cudaFreeHost(h->status_host);
  if (h->host_exec) cudaGraphExecDestroy(h->host_exec);
  if (h->capture_stream) cudaStreamDestroy(h->capture_stream);
  cudaSetDevice(current);
  delete h;
}

// Copy a weight array to the device when it lives in host memory.
int stage_input(const void* src, size_t bytes, const uint8_t** dev, std::vector<void*>& temps) {
  if (is_device_pointer(src)) {
    *dev = static_cast<const uint8_t*>(src);
    return MOE_OK;
  }
  void* p = nullptr;
  MOE_CUDA(cudaMalloc(&p, bytes));
  temps.push_back(p);
  MOE_CUDA(cudaMemcpy(p, src, bytes, cudaMemcpyHostToDevice));
  *dev = static_cast<const uint8_t*>(p);
  return MOE_OK;
}

int build_handle(moe_ctx* h, const void* w13, const void* s13, const void* w2, const void* s2) {
  const Geometry& g = h->g;
  cudaDeviceProp prop{};
  MOE_CUDA(cudaGetDevice(&h->device));
  MOE_CUDA(cudaGetDeviceProperties(&prop, h->device));
  h->smem_bytes = moe::experts_max_smem_bytes(g);
  if (!moe::experts_layout_aligned(g)) {
    std::snprintf(g_detail, sizeof g_detail, "internal: misaligned shared-memory layout");
    return MOE_ERR_UNSUPPORTED;
  }
  if (moe_device_supported(prop.major, prop.minor, prop.sharedMemPerBlockOptin) != MOE_OK) {
    std::snprintf(g_detail, sizeof g_detail,
                  "needs an sm_103 GPU (GB300) with %d B of shared memory per block; found sm_%d%d "
                  "with %zu B (the library carries sm_103a code only)",
                  moe::experts_max_smem_bytes(moe::make_geometry(1, 256, MOE_MAX_INTER)), prop.major,
                  prop.minor, static_cast<size_t>(prop.sharedMemPerBlockOptin));
    return MOE_ERR_UNSUPPORTED;
  }
  h->sms = prop.multiProcessorCount;
  MOE_CUDA(cudaDeviceGetAttribute(&h->host_atomics, cudaDevAttrHostNativeAtomicSupported, h->device));
  MOE_CUDA(moe::experts_configure(g));
  int per_sm = 0;
  MOE_CUDA(moe::experts_occupancy(g, &per_sm));
  if (per_sm < 1) {
    std::snprintf(g_detail, sizeof g_detail, "experts kernel does not fit on an SM");
    return MOE_ERR_UNSUPPORTED;
  }
  h->grid = h->sms < moe::kMaxGrid ? h->sms : moe::kMaxGrid;  // one co-resident CTA per SM
  for (int b = 1; b <= moe::kSmallMaxBatch; ++b) h->small_ok[b] = moe::small_fits(g, b, h->grid) ? 1 : 0;

  // Weights: one 17 KB block per stage.
  h->stage_bytes = static_cast<size_t>(g.E) * g.SPE * moe::kStageBytes;
  MOE_CUDA(cudaMalloc(&h->stages, h->stage_bytes));
  std::vector<void*> temps;
  const uint8_t *d13, *ds13, *d2, *ds2;
  const size_t n13 = static_cast<size_t>(g.E) * 2 * g.I * (g.H / 2);
  const size_t n2 = static_cast<size_t>(g.E) * g.H * (g.I / 2);
  int rc = stage_input(w13, n13, &d13, temps);
  if (rc == MOE_OK) rc = stage_input(s13, n13 / 16, &ds13, temps);
  if (rc == MOE_OK) rc = stage_input(w2, n2, &d2, temps);
  if (rc == MOE_OK) rc = stage_input(s2, n2 / 16, &ds2, temps);
  if (rc == MOE_OK) {
    cudaError_t e = moe::launch_repack(d13, ds13, d2, ds2, g, h->stages, nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) rc = cuda_fail(e, "weight repack");
  }
  for (void* p : temps) cudaFree(p);
  if (rc != MOE_OK) return rc;

  // Plan, unit table and workspace in one allocation.
  h->unit_cap = moe::unit_capacity(MOE_MAX_BATCH, g.E);
  const size_t sizes[] = {
      static_cast<size_t>(MOE_MAX_BATCH) * g.H,                 // plan codes
      static_cast<size_t>(MOE_MAX_BATCH) * (g.H / moe::kBlock), // plan scales
      8,                                                        // unit count, pair count
      static_cast<size_t>(h->unit_cap) * 4,                     // unit experts
      static_cast<size_t>(h->unit_cap) * moe::kUnitRows * 2,    // unit rows
      static_cast<size_t>(h->unit_cap) * g.P1 * 4,              // FC1 item counters
      static_cast<size_t>(h->unit_cap) * g.KC2 * 4,             // hidden flags
      static_cast<size_t>(h->grid) * 2 * 2 * 16 * moe::kTileM * 4,  // partials (16-row units)
      static_cast<size_t>(h->unit_cap) * g.hidden_bytes,        // hidden images
      4,                                                        // status
      static_cast<size_t>(MOE_MAX_BATCH) * MOE_TOPK,            // kept pairs
      static_cast<size_t>(MOE_MAX_BATCH) * MOE_TOPK * g.H * 2,  // staged per-pair rows
      static_cast<size_t>(moe::kMaxSpanCtas) * 2 * 8,           // launch clock
      moe::small_reader_bytes(g),                               // small-batch read counts
      static_cast<size_t>(h->unit_cap) * 4,                     // pairs of units
      moe::small_piece_bytes(g),                                // small-batch segment slots
      moe::kSmallCounterBytes,                                  // small-batch claim counters
      16,                                                       // early start: ready, arrive, passed
  };
  size_t offsets[18], total = 0;
  for (int i = 0; i < 18; ++i) {
    offsets[i] = total;
    total += round256(sizes[i]);
  }
  h->workspace_bytes = total;
  MOE_CUDA(cudaMalloc(&h->workspace, total));
  MOE_CUDA(cudaMemset(h->workspace, 0, total));
  uint8_t* w = h->workspace;
  h->plan_codes = w + offsets[0];
  h->plan_scales = w + offsets[1];
  h->unit_count = reinterpret_cast<int32_t*>(w + offsets[2]);
  h->unit_expert = reinterpret_cast<int32_t*>(w + offsets[3]);
  h->unit_rows = reinterpret_cast<int16_t*>(w + offsets[4]);
  h->item_counters = reinterpret_cast<uint32_t*>(w + offsets[5]);
  h->hidden_flags = reinterpret_cast<uint32_t*>(w + offsets[6]);
  h->partials = reinterpret_cast<float*>(w + offsets[7]);
  h->hidden = w + offsets[8];
  h->status = reinterpret_cast<int32_t*>(w + offsets[9]);
  h->pair_kept = w + offsets[10];
  h->staged = reinterpret_cast<uint16_t*>(w + offsets[11]);
  h->span = reinterpret_cast<uint64_t*>(w + offsets[12]);
  h->piece_readers = reinterpret_cast<uint32_t*>(w + offsets[13]);
  h->wide_units = reinterpret_cast<uint32_t*>(w + offsets[14]);
  h->piece_sums = reinterpret_cast<uint32_t*>(w + offsets[15]);
  h->small_counters = reinterpret_cast<uint32_t*>(w + offsets[16]);
  h->ready = reinterpret_cast<uint32_t*>(w + offsets[17]);
  h->arrive = h->ready + 1;
  h->passed = h->ready + 2;
  MOE_CUDA(cudaMemset(h->piece_sums, 0xFF, moe::small_piece_bytes(g)));  // every word the sentinel
  MOE_CUDA(cudaMallocHost(&h->status_host, 4));
  h->status_dev = h->status;
  return encode_weight_map(h);
}

moe::PrepArgs prep_args(moe_ctx* h, const void* x, const int32_t* ids, int batch, int roles) {
  moe::PrepArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.ids = ids;
  a.B = batch;
  a.H = h->g.H;
  a.E = h->g.E;
  a.P1 = h->g.P1;
  a.KC2 = h->g.KC2;
  a.unit_cap = h->unit_cap;
  a.plan_codes = h->plan_codes;
  a.plan_scales = h->plan_scales;
  a.unit_count = h->unit_count;
  a.unit_expert = h->unit_expert;
  a.unit_rows = h->unit_rows;
  a.wide_units = h->wide_units;
  a.item_counters = h->item_counters;
  a.hidden_flags = h->hidden_flags;
  a.pair_kept = h->pair_kept;
  a.status = h->status_dev;
  a.roles = roles;
  a.quant_blocks = moe::prep_quant_blocks(batch, h->g.H);
  return a;
}

int check_batch(int batch) { return (batch >= 1 && batch <= MOE_MAX_BATCH) ? MOE_OK : MOE_ERR_ARG; }

// The handle whose call was the last this library launched on each stream.
// A grid call that follows another handle's call on its stream starts early:
// its prep grid writes this handle's tables (nothing the previous call
// touches) without waiting for the previous grid, and its experts kernel
// streams FC1 as soon as its CTAs are resident, waiting for the previous
// grid only before its first output row. Every kernel of this library waits
// for the grid before it ahead of ending, and lets the next launch start only
// after that wait, so when an early prep grid starts, the call before the
// previous one on the stream (possibly this handle's last) has ended.
// `overlaps`: the call's last launch lets the next one start while it still
// runs (moe_run, moe_run_noalloc), so the next call's CTAs start one by one
// as its CTAs leave, and an early grid call skews its FC1 split to match.
struct LastLaunch {
  const moe_ctx* h;
  bool overlaps;
};
std::mutex g_stream_mutex;
std::unordered_map<cudaStream_t, LastLaunch> g_last_launch;

// Whether this call follows another handle's call on `s` (early start), and
// whether that call's last launch overlaps this one; records this call.
bool follows_other_handle(const moe_ctx* h, cudaStream_t s, bool* prev_overlaps) {
  std::lock_guard<std::mutex> lock(g_stream_mutex);
  auto it = g_last_launch.find(s);
  const bool other = it != g_last_launch.end() && it->second.h != h;
  *prev_overlaps = other && it->second.overlaps;
  g_last_launch[s] = LastLaunch{h, true};
  return other;
}

void note_launch(const moe_ctx* h, cudaStream_t s, bool overlaps = false) {
  std::lock_guard<std::mutex> lock(g_stream_mutex);
  g_last_launch[s] = LastLaunch{h, overlaps};
}

// A handle's buffers, tensor map and kernels belong to the device that was
// current at moe_prepare: every call that launches, copies or synchronizes
// refuses to run with another device current.
int check_device(const moe_ctx* h) {
  int current = -1;
  MOE_CUDA(cudaGetDevice(&current));
  if (current != h->device) {
    std::snprintf(g_detail, sizeof g_detail,
                  "handle prepared on device %d used with device %d current", h->device, current);
    return MOE_ERR_ARG;
  }
  return MOE_OK;
}

#define MOE_CHECK_DEVICE(h)                     \
  do {                                          \
    const int moe_rc_ = check_device(h);        \
    if (moe_rc_ != MOE_OK) return moe_rc_;      \
  } while (0)

// Whether a call of `batch` tokens with its routing ids runs on the
// small-batch kernel alone (no prep grid).
bool small_call(const moe_ctx* h, int batch) {
  return batch <= moe::kSmallMaxBatch && moe::small_path_serves(h->path, batch) && h->small_ok[batch];
}

// ids: the call's routing ids when the same call's prep grid runs just
// before on this stream (or, x given, when the call is the small-batch kernel
// alone), else null.
int launch_experts(moe_ctx* h, void* out, int batch, const int32_t* ids, cudaStream_t stream,
                   const void* x = nullptr, bool early = false, bool skew = false) {
  moe::ExpertsArgs a{};
  a.skew = skew ? 1 : 0;
  if (early) {
    a.early = 1;
    a.seq = h->seq;
    a.ready = h->ready;
    a.passed = h->passed;
  }
  a.wmap = h->wmap;
  a.stages = h->stages;
  a.ids = ids;
  a.plan_codes = h->plan_codes;
  a.plan_scales = h->plan_scales;
  a.unit_count = h->unit_count;
  a.unit_expert = h->unit_expert;
  a.unit_rows = h->unit_rows;
  a.wide_units = h->wide_units;
  a.item_counters = h->item_counters;
  a.hidden_flags = h->hidden_flags;
  a.partials = h->partials;
  a.hidden = h->hidden;
  a.out = static_cast<uint16_t*>(out);
  a.status = h->status_dev;
  a.B = batch;
  a.g = h->g;
  a.timeout_ns = h->timeout_ns;
  a.withhold_unit = h->withhold;
  a.withhold_image = h->withhold_image;
  a.span = h->span_on ? h->span : nullptr;
  a.trace = h->trace;
  a.x = static_cast<const uint16_t*>(x);
  a.piece_sums = h->piece_sums;
  a.piece_readers = h->piece_readers;
  a.small_counters = h->small_counters;
  a.seg_cap = moe::small_seg_cap(h->g);
  a.piece_words = moe::kSmallPieceWords;
  // Consecutive small-batch calls take alternate halves of that kernel's
  // slots and counters.
  a.parity = h->small_parity;
  const bool small = ids != nullptr && small_call(h, batch);
  if (small) h->small_parity ^= 1;
  a.pair_kept = h->pair_kept;
  MOE_CUDA(moe::launch_experts(a, h->grid, stream, true, h->path, small));
  return MOE_OK;
}

// moe_run; fused = false keeps the prep grid in front of the small-batch
// kernel (for inputs in host memory, which the prep grid reads once).
int run_call(moe_handle h, const void* x_bf16, const int32_t* topk_ids, void* out_bf16, int batch,
             void* stream, bool fused) {
  if (h == nullptr || !x_bf16 || !topk_ids || !out_bf16) return MOE_ERR_ARG;
  if (!aligned16(x_bf16) || !aligned16(topk_ids) || !aligned16(out_bf16) || check_batch(batch))
    return MOE_ERR_ARG;
  MOE_CHECK_DEVICE(h);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int rc;
  if (fused && small_call(h, batch)) {
    // One launch: the small-batch kernel quantizes x and groups the ids itself.
    note_launch(h, s, true);
    rc = launch_experts(h, out_bf16, batch, topk_ids, s, x_bf16);
  } else {
    // The persistent grid kernel may start early after another handle's call.
    const bool grid = !small_call(h, batch) && moe_kernel_path(h, batch) == moe::kPathGrid;
    bool prev_overlaps = false;
    const bool early = follows_other_handle(h, s, &prev_overlaps) && grid && fused;
    moe::PrepArgs pa = prep_args(h, x_bf16, topk_ids, batch, moe::kPrepQuantize | moe::kPrepGroup);
    pa.chained = 1;
    if (early) {
      pa.early = 1;
      pa.seq = ++h->seq;
      pa.ready = h->ready;
      pa.arrive = h->arrive;
    }
    MOE_CUDA(moe::launch_prep(pa, s));
    rc = launch_experts(h, out_bf16, batch, topk_ids, s, nullptr, early, early && prev_overlaps);
  }
  if (rc != MOE_OK) return rc;
  h->plan_batch = batch;
  h->group_batch = batch;
  h->grouped = 1;
  h->ran = 1;
  return MOE_OK;
}

// Captures moe_run on host buffers, with the kernels reporting into the
// pinned status word, into the handle's replay graph.
int capture_host_run(moe_ctx* h, const void* x_host, const int32_t* ids_host, void* out_host,
                     int batch) {
  if (h->host_exec) {
    cudaGraphExecDestroy(h->host_exec);
    h->host_exec = nullptr;
  }
  if (h->capture_stream == nullptr)
    MOE_CUDA(cudaStreamCreateWithFlags(&h->capture_stream, cudaStreamNonBlocking));
  MOE_CUDA(cudaStreamBeginCapture(h->capture_stream, cudaStreamCaptureModeThreadLocal));
  h->status_dev = h->status_host;
  const int rc = run_call(h, x_host, ids_host, out_host, batch, h->capture_stream, false);
  h->status_dev = h->status;
  cudaGraph_t graph = nullptr;
  const cudaError_t ce = cudaStreamEndCapture(h->capture_stream, &graph);
  if (rc != MOE_OK) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  MOE_CUDA(ce);
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  MOE_CUDA(ie);
  h->host_exec = exec;
  h->host_x = x_host;
  h->host_ids = ids_host;
  h->host_out = out_host;
  h->host_batch = batch;
  h->host_settings = h->settings;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_prepare(moe_handle* out, const void* w13, const void* s13, const void* w2, const void* s2,
                int experts, int hidden, int inter) {
  if (out == nullptr) return MOE_ERR_ARG;
  *out = nullptr;
  if (!w13 || !s13 || !w2 || !s2) return MOE_ERR_ARG;
  if (experts < 1 || experts > MOE_MAX_EXPERTS) return MOE_ERR_ARG;
  if (hidden < 256 || hidden > MOE_MAX_HIDDEN || hidden % 256 != 0) return MOE_ERR_ARG;
  if (inter < 32 || inter > MOE_MAX_INTER || inter % 32 != 0) return MOE_ERR_ARG;
  moe_ctx* h = new (std::nothrow) moe_ctx();
  if (h == nullptr) return MOE_ERR_CUDA;
  h->g = moe::make_geometry(experts, hidden, inter);
  const int rc = build_handle(h, w13, s13, w2, s2);
  if (rc != MOE_OK) {
    release(h);
    return rc;
  }
  *out = h;
  return MOE_OK;
}

int moe_quantize(moe_handle h, const void* x_bf16, int batch, void* stream) {
  if (h == nullptr || x_bf16 == nullptr || !aligned16(x_bf16) || check_batch(batch)) return MOE_ERR_ARG;
  MOE_CHECK_DEVICE(h);
  note_launch(h, static_cast<cudaStream_t>(stream));
  MOE_CUDA(moe::launch_prep(prep_args(h, x_bf16, nullptr, batch, moe::kPrepQuantize),
                            static_cast<cudaStream_t>(stream)));
  h->plan_batch = batch;
  return MOE_OK;
}

int moe_group(moe_handle h, const int32_t* topk_ids, int batch, void* stream) {
  if (h == nullptr || topk_ids == nullptr || !aligned16(topk_ids) || check_batch(batch))
    return MOE_ERR_ARG;
  MOE_CHECK_DEVICE(h);
  note_launch(h, static_cast<cudaStream_t>(stream));
  MOE_CUDA(moe::launch_prep(prep_args(h, nullptr, topk_ids, batch, moe::kPrepGroup),
                            static_cast<cudaStream_t>(stream)));
  h->grouped = 1;
  h->group_batch = batch;
  return MOE_OK;
}

int moe_run(moe_handle h, const void* x_bf16, const int32_t* topk_ids, void* out_bf16, int batch,
            void* stream) {
  return run_call(h, x_bf16, topk_ids, out_bf16, batch, stream, true);
}

int moe_run_combined(moe_handle h, const void* x_bf16, const int32_t* topk_ids,
                     const float* topk_weights, void* out_bf16, int batch, void* stream) {
  if (h == nullptr || !x_bf16 || !topk_ids || !topk_weights || !out_bf16) return MOE_ERR_ARG;
  if (!aligned16(x_bf16) || !aligned16(topk_ids) || !aligned16(topk_weights) ||
      !aligned16(out_bf16) || check_batch(batch))
    return MOE_ERR_ARG;
  MOE_CHECK_DEVICE(h);
  const int rc = run_call(h, x_bf16, topk_ids, h->staged, batch, stream, true);
  if (rc != MOE_OK) return rc;
  moe::CombineArgs c{};
  c.rows = h->staged;
  c.weights = topk_weights;
  c.kept = h->pair_kept;
  c.out = static_cast<uint16_t*>(out_bf16);
  c.B = batch;
  c.H = h->g.H;
  MOE_CUDA(moe::launch_combine(c, static_cast<cudaStream_t>(stream)));
  note_launch(h, static_cast<cudaStream_t>(stream));  // the combine lets nothing start early
  return MOE_OK;
}

int moe_experts(moe_handle h, void* out_bf16, int batch, void* stream) {
  if (h == nullptr || out_bf16 == nullptr || !aligned16(out_bf16) || check_batch(batch))
    return MOE_ERR_ARG;
  MOE_CHECK_DEVICE(h);
  note_launch(h, static_cast<cudaStream_t>(stream));
  if (h->plan_batch != batch || h->group_batch != batch) return MOE_ERR_STATE;
  const int rc = launch_experts(h, out_bf16, batch, nullptr, static_cast<cudaStream_t>(stream));
  if (rc == MOE_OK) h->ran = 1;
  return rc;
}

int moe_sync_status(moe_handle h, void* stream) {
  if (h == nullptr) return MOE_ERR_ARG;
  MOE_CHECK_DEVICE(h);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_CUDA(cudaMemcpyAsync(h->status_host, h->status, 4, cudaMemcpyDeviceToHost, s));
  MOE_CUDA(cudaMemsetAsync(h->status, 0, 4, s));
  MOE_CUDA(cudaStreamSynchronize(s));
  const int status = *h->status_host;
  if (status == MOE_ERR_DEVICE_TIMEOUT) {
    // A bounded wait ran out, so some segment slots of the small-batch
    // kernel may not have been read by all their consumers (and put back to
    // rest), and its claim counters may not be back at zero: reset them.
    MOE_CUDA(cudaMemsetAsync(h->piece_readers, 0, moe::small_reader_bytes(h->g), s));
    MOE_CUDA(cudaMemsetAsync(h->piece_sums, 0xFF, moe::small_piece_bytes(h->g), s));
    MOE_CUDA(cudaMemsetAsync(h->small_counters, 0, moe::kSmallCounterBytes, s));
    // An early-start call may have stopped before its flag went back to rest.
    MOE_CUDA(cudaMemsetAsync(h->ready, 0, 3 * sizeof(uint32_t), s));
    MOE_CUDA(cudaStreamSynchronize(s));
  }
  return status;
}

bool is_pinned_host(const void* p) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return attr.type == cudaMemoryTypeHost && attr.devicePointer == p;
}

int moe_run_host(moe_handle h, const void* x_host, const int32_t* ids_host, void* out_host,
                 int batch, void* stream) {
  if (h == nullptr || !x_host || !ids_host || !out_host || check_batch(batch)) return MOE_ERR_ARG;
  MOE_CHECK_DEVICE(h);
  note_launch(h, static_cast<cudaStream_t>(stream));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (h->host_atomics && aligned16(x_host) && aligned16(ids_host) && aligned16(out_host) &&
      is_pinned_host(x_host) && is_pinned_host(ids_host) && is_pinned_host(out_host)) {
    // Pinned buffers are mapped into the GPU's address space (the same
    // pointers; coherent over the GPU-CPU link): the prep grid reads x and ids
    // from them, the epilogue writes the rows into them, and the kernels
    // report into a pinned status word, so the call makes no copies at all.
    // The two launches are captured into a graph on first use (and again
    // when the buffers, the batch or a setting change); each call is then a
    // single graph launch.
    *reinterpret_cast<volatile int32_t*>(h->status_host) = 0;
    if (h->host_exec == nullptr || h->host_x != x_host || h->host_ids != ids_host ||
        h->host_out != out_host || h->host_batch != batch || h->host_settings != h->settings) {
      const int rc = capture_host_run(h, x_host, ids_host, out_host, batch);
      if (rc != MOE_OK) return rc;
    }
    MOE_CUDA(cudaGraphLaunch(h->host_exec, s));
    h->plan_batch = batch;  // what moe_run records, for the read-back calls
    h->group_batch = batch;
    h->grouped = 1;
    h->ran = 1;
    MOE_CUDA(cudaStreamSynchronize(s));
    return *reinterpret_cast<volatile int32_t*>(h->status_host);
  }
  const size_t xb = round256(static_cast<size_t>(MOE_MAX_BATCH) * h->g.H * 2);
  const size_t ib = round256(static_cast<size_t>(MOE_MAX_BATCH) * MOE_TOPK * 4);
  const size_t ob = static_cast<size_t>(MOE_MAX_BATCH) * MOE_TOPK * h->g.H * 2;
  if (h->io == nullptr) MOE_CUDA(cudaMalloc(&h->io, xb + ib + ob));
  uint8_t* dx = h->io;
  int32_t* dids = reinterpret_cast<int32_t*>(h->io + xb);
  uint8_t* dout = h->io + xb + ib;
  const size_t x_bytes = static_cast<size_t>(batch) * h->g.H * 2;
  const size_t ids_bytes = static_cast<size_t>(batch) * MOE_TOPK * 4;
  const size_t out_bytes = static_cast<size_t>(batch) * MOE_TOPK * h->g.H * 2;
  MOE_CUDA(cudaMemcpyAsync(dx, x_host, x_bytes, cudaMemcpyHostToDevice, s));
  MOE_CUDA(cudaMemcpyAsync(dids, ids_host, ids_bytes, cudaMemcpyHostToDevice, s));
  const int rc = moe_run(h, dx, dids, dout, batch, stream);
  if (rc != MOE_OK) return rc;
  MOE_CUDA(cudaMemcpyAsync(out_host, dout, out_bytes, cudaMemcpyDeviceToHost, s));
  return moe_sync_status(h, stream);
}

int moe_copy_plan(moe_handle h, uint8_t* codes, uint8_t* scales, int batch) {
  if (h == nullptr || codes == nullptr || scales == nullptr) return MOE_ERR_ARG;
  MOE_CHECK_DEVICE(h);
  if (h->plan_batch == 0) return MOE_ERR_STATE;
  if (batch < 1 || batch > h->plan_batch) return MOE_ERR_ARG;
  MOE_CUDA(cudaDeviceSynchronize());
  MOE_CUDA(cudaMemcpy(codes, h->plan_codes, static_cast<size_t>(batch) * h->g.H,
                      cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemcpy(scales, h->plan_scales, static_cast<size_t>(batch) * (h->g.H / moe::kBlock),
                      cudaMemcpyDeviceToHost));
  return MOE_OK;
}

int moe_copy_units(moe_handle h, int32_t* count, int32_t* experts, int16_t* rows, int capacity) {
  if (h == nullptr || count == nullptr) return MOE_ERR_ARG;
  MOE_CHECK_DEVICE(h);
  if (!h->grouped) return MOE_ERR_STATE;
  MOE_CUDA(cudaDeviceSynchronize());
  MOE_CUDA(cudaMemcpy(count, h->unit_count, 4, cudaMemcpyDeviceToHost));
  if (*count > capacity || (*count > 0 && (experts == nullptr || rows == nullptr))) return MOE_ERR_ARG;
  if (*count > 0) {
    MOE_CUDA(cudaMemcpy(experts, h->unit_expert, static_cast<size_t>(*count) * 4,
                        cudaMemcpyDeviceToHost));
    MOE_CUDA(cudaMemcpy(rows, h->unit_rows, static_cast<size_t>(*count) * moe::kUnitRows * 2,
                        cudaMemcpyDeviceToHost));
  }
  return MOE_OK;
}

int moe_copy_hidden(moe_handle h, uint8_t* codes, uint8_t* scales, int units) {
  if (h == nullptr || codes == nullptr || scales == nullptr || units < 0) return MOE_ERR_ARG;
  MOE_CHECK_DEVICE(h);
  if (!h->ran) return MOE_ERR_STATE;
  if (units > h->unit_cap) return MOE_ERR_ARG;
  const Geometry& g = h->g;
  std::vector<uint8_t> img(static_cast<size_t>(units) * g.hidden_bytes);
  MOE_CUDA(cudaDeviceSynchronize());
  if (!img.empty())
    MOE_CUDA(cudaMemcpy(img.data(), h->hidden, img.size(), cudaMemcpyDeviceToHost));
  for (int u = 0; u < units; ++u) {
    const uint8_t* base = img.data() + static_cast<size_t>(u) * g.hidden_bytes;
    for (int r = 0; r < moe::kUnitRows; ++r) {
      for (int j = 0; j < g.I; ++j) {
        const int c = j / moe::kChunkK, k = j % moe::kChunkK;
        codes[(static_cast<size_t>(u) * moe::kUnitRows + r) * g.I + j] =
            base[c * moe::kActImageBytes + moe::swizzle128(r, k >> 4) + (k & 15)];
      }
      for (int b = 0; b < g.I / moe::kBlock; ++b) {
        const int c = b / 4, kb = b % 4;
        scales[(static_cast<size_t>(u) * moe::kUnitRows + r) * (g.I / moe::kBlock) + b] =
            base[g.KC2 * moe::kActImageBytes + c * moe::kScaleAtomBytes + moe::scale_atom(r, kb)];
      }
    }
  }
  return MOE_OK;
}

int moe_set_timeout(moe_handle h, uint64_t nanoseconds) {
  if (h == nullptr) return MOE_ERR_ARG;
  h->timeout_ns = nanoseconds ? nanoseconds : 2000000000ull;
  ++h->settings;
  return MOE_OK;
}

int moe_debug_withhold(moe_handle h, int unit) {
  if (h == nullptr || unit < -1) return MOE_ERR_ARG;
  h->withhold = unit;
  ++h->settings;
  return MOE_OK;
}

int moe_debug_withhold_image(moe_handle h, int unit) {
  if (h == nullptr || unit < -1) return MOE_ERR_ARG;
  h->withhold_image = unit;
  ++h->settings;
  return MOE_OK;
}

int moe_debug_paths(moe_handle h, int path) {
  if (h == nullptr || path < moe::kPathGrid || path > moe::kPathSmallWide) return MOE_ERR_ARG;
  h->path = path;
  ++h->settings;
  return MOE_OK;
}

int moe_debug_kernel_span(moe_handle h, int enable) {
  if (h == nullptr || enable < 0 || enable > 1) return MOE_ERR_ARG;
  MOE_CHECK_DEVICE(h);
  if (enable && !h->span_on) {
    MOE_CUDA(cudaDeviceSynchronize());
    MOE_CUDA(cudaMemset(h->span, 0, static_cast<size_t>(moe::kMaxSpanCtas) * 2 * 8));
  }
  h->span_on = enable;
  ++h->settings;
  return MOE_OK;
}

int moe_read_kernel_span(moe_handle h, uint64_t* span_ns) {
  if (h == nullptr || span_ns == nullptr) return MOE_ERR_ARG;
  MOE_CHECK_DEVICE(h);
  std::vector<uint64_t> words(static_cast<size_t>(moe::kMaxSpanCtas) * 2);
  MOE_CUDA(cudaDeviceSynchronize());
  MOE_CUDA(cudaMemcpy(words.data(), h->span, words.size() * 8, cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemset(h->span, 0, words.size() * 8));
  uint64_t first = ~0ull, last = 0;
  for (size_t c = 0; c < words.size() / 2; ++c) {
    if (words[2 * c] == 0) continue;  // no CTA of that index in the last launch
    if (words[2 * c] < first) first = words[2 * c];
    if (words[2 * c + 1] > last) last = words[2 * c + 1];
  }
  if (first == ~0ull || last < first) return MOE_ERR_STATE;
  *span_ns = last - first;
  return MOE_OK;
}

#ifdef MOE_TRACE
// Trace builds only: per-CTA phase stamps (16 words per CTA) into `buffer`.
int moe_debug_trace(moe_handle h, void* buffer) {
  if (h == nullptr) return MOE_ERR_ARG;
  h->trace = static_cast<uint64_t*>(buffer);
  ++h->settings;
  return MOE_OK;
}
#endif

int moe_cluster_size(moe_handle h, int batch) {
  if (h == nullptr || check_batch(batch)) return -MOE_ERR_ARG;
  return h->path == moe::kPathCluster ? moe::cluster_size_for(h->g, batch) : 0;
}

int moe_kernel_path(moe_handle h, int batch) {
  if (h == nullptr || check_batch(batch)) return -MOE_ERR_ARG;
  if (small_call(h, batch)) return moe::kPathSmall;
  if (h->path == moe::kPathCluster && moe::cluster_size_for(h->g, batch) > 0) return moe::kPathCluster;
  return moe::kPathGrid;
}

int moe_info(moe_handle h, moe_info_t* info) {
  if (h == nullptr || info == nullptr) return MOE_ERR_ARG;
  info->experts = h->g.E;
  info->hidden = h->g.H;
  info->inter = h->g.I;
  info->hidden_floor_rule = h->g.floor_rule;
  info->grid = h->grid;
  info->ring_stages = moe::kRingStages;
  info->smem_bytes = h->smem_bytes;
  info->stages_per_expert = h->g.SPE;
  info->unit_capacity = h->unit_cap;
  info->hidden_image_bytes = h->g.hidden_bytes;
  info->weight_bytes = h->stage_bytes;
  info->workspace_bytes = h->workspace_bytes;
  return MOE_OK;
}

void moe_destroy(moe_handle h) { release(h); }

const char* moe_error_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported device or configuration";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_IDS: return "expert id out of range or repeated within a token";
    case MOE_ERR_STATE: return "call order: the data asked for was not produced yet";
    default: return "unknown status";
  }
}

const char* moe_last_error_detail(void) { return g_detail; }

int moe_small_batch_build(int experts, int hidden, int inter, int batch, int grid) {
  if (experts < 1 || experts > MOE_MAX_EXPERTS) return -MOE_ERR_ARG;
  if (hidden < 256 || hidden > MOE_MAX_HIDDEN || hidden % 256 != 0) return -MOE_ERR_ARG;
  if (inter < 32 || inter > MOE_MAX_INTER || inter % 32 != 0) return -MOE_ERR_ARG;
  if (batch < 1 || batch > moe::kSmallMaxBatch || grid < 1 || grid > moe::kMaxGrid) return -MOE_ERR_ARG;
  return moe::small_build(moe::make_geometry(experts, hidden, inter), batch, grid);
}

int moe_device_supported(int cc_major, int cc_minor, size_t smem_per_block_optin) {
  if (cc_major != 10 || cc_minor != 3) return MOE_ERR_UNSUPPORTED;
  const size_t need = static_cast<size_t>(moe::experts_max_smem_bytes(moe::make_geometry(1, 256, MOE_MAX_INTER)));
  return smem_per_block_optin >= need ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// moe_run without allocation (no counterpart on the pages).
//
// Some callers cannot call cudaMalloc when they run a layer: a runtime that
// hands all device memory to its own pool at start-up, or code that must not
// allocate on the decode path. moe_run itself allocates nothing either, but
// its scratch lives in the handle's workspace, which is sized for the largest
// batch. moe_run_noalloc runs the same two kernels with every per-call
// scratch buffer (activation plan, unit table, split-K counters and partial
// sums, hidden-vector images) carved out of one fixed, module-scope device
// array instead; the caller still passes x, ids and out, and the handle still
// supplies the prepared weights.

namespace {

// Scratch shared by every moe_run_noalloc call on a device. Every GPU that
// loads this library holds it until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch per device. In host code the array's
// name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, once per device, with that device current.
constexpr int kNoallocDevices = 64;
void* g_noalloc_address[kNoallocDevices] = {};
std::mutex g_noalloc_mutex;

int noalloc_scratch(int device, uint8_t** base) {
  if (device < 0 || device >= kNoallocDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_address[device] == nullptr) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_noalloc_address[device] = ptr;
  }
  *base = static_cast<uint8_t*>(g_noalloc_address[device]);
  return MOE_OK;
}

}  // namespace

extern "C" int moe_run_noalloc(moe_handle h, const void* x_bf16, const int32_t* topk_ids,
                               void* out_bf16, int batch, void* stream) {
  if (h == nullptr || !x_bf16 || !topk_ids || !out_bf16) return MOE_ERR_ARG;
  if (!aligned16(x_bf16) || !aligned16(topk_ids) || !aligned16(out_bf16) || check_batch(batch))
    return MOE_ERR_ARG;
  const Geometry& g = h->g;
  const int cap = moe::unit_capacity(batch, g.E);
  // Here the small-batch kernel serves one or two tokens (its segment slots
  // then hold two rows each: a smaller share of the static buffer).
  const bool small = batch <= 2 && small_call(h, batch);
  const int small_cap = 2 * MOE_TOPK * g.P1 * moe::small_spi(g.KC1), small_words = 2 * 2 * moe::kTileM;
  const size_t sizes[] = {
      static_cast<size_t>(batch) * g.H,                            // plan codes
      static_cast<size_t>(batch) * (g.H / moe::kBlock),            // plan scales
      8,                                                           // unit count, pair count
      static_cast<size_t>(cap) * 4,                                // unit experts
      static_cast<size_t>(cap) * moe::kUnitRows * 2,               // unit rows
      static_cast<size_t>(cap) * g.P1 * 4,                         // FC1 item counters
      static_cast<size_t>(cap) * g.KC2 * 4,                        // hidden flags
      static_cast<size_t>(h->grid) * 2 * 2 * (batch > moe::kUnitRows ? 16 : 8) * moe::kTileM * 4,  // partials
      static_cast<size_t>(cap) * g.hidden_bytes,                   // hidden images
      small ? static_cast<size_t>(small_cap) * 4 : 0,             // small-batch read counts (one half)
      static_cast<size_t>(cap) * 4,                                // pairs of units
      small ? static_cast<size_t>(small_cap) * small_words * 4 : 0,  // small-batch segment slots (one half)
      small ? moe::kSmallCounterBytes : 0,                         // small-batch claim counters
  };
  size_t offsets[13], total = 0;
  for (int i = 0; i < 13; ++i) {
    offsets[i] = total;
    total += round256(sizes[i]);
  }
  if (total > MOE_NOALLOC_SCRATCH_BYTES) {
    std::snprintf(g_detail, sizeof g_detail,
                  "moe_run_noalloc: batch %d of this layer needs %zu bytes of scratch, more than "
                  "the %d-byte static buffer",
                  batch, total, MOE_NOALLOC_SCRATCH_BYTES);
    return MOE_ERR_ARG;
  }
  MOE_CHECK_DEVICE(h);
  uint8_t* w = nullptr;
  const int rc = noalloc_scratch(h->device, &w);
  if (rc != MOE_OK) return rc;

  // The grouping block of the prep kernel clears the counters and flags the
  // grid kernel needs at zero; the small-batch kernel's piece slots and read
  // counts are put to rest below. Every other scratch byte is written before
  // it is read within the call, so nothing is left over from the last call.
  moe::PrepArgs pa = prep_args(h, x_bf16, topk_ids, batch, moe::kPrepQuantize | moe::kPrepGroup);
  pa.unit_cap = cap;
  pa.plan_codes = w + offsets[0];
  pa.plan_scales = w + offsets[1];
  pa.unit_count = reinterpret_cast<int32_t*>(w + offsets[2]);
  pa.unit_expert = reinterpret_cast<int32_t*>(w + offsets[3]);
  pa.unit_rows = reinterpret_cast<int16_t*>(w + offsets[4]);
  pa.wide_units = reinterpret_cast<uint32_t*>(w + offsets[10]);
  pa.item_counters = reinterpret_cast<uint32_t*>(w + offsets[5]);
  pa.hidden_flags = reinterpret_cast<uint32_t*>(w + offsets[6]);
  pa.pair_kept = nullptr;  // only the combine reads these flags, and this call has no combine
  pa.chained = 1;          // this call's experts kernel follows at once
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  note_launch(h, s, true);
  uint32_t* piece_readers = reinterpret_cast<uint32_t*>(w + offsets[9]);
  uint32_t* piece_sums = reinterpret_cast<uint32_t*>(w + offsets[11]);
  uint32_t* small_counters = reinterpret_cast<uint32_t*>(w + offsets[12]);
  if (small) {  // memsets, not allocations; the call takes half 0 of the slots
    MOE_CUDA(cudaMemsetAsync(piece_readers, 0, static_cast<size_t>(small_cap) * 4, s));
    MOE_CUDA(cudaMemsetAsync(piece_sums, 0xFF, static_cast<size_t>(small_cap) * small_words * 4, s));
    MOE_CUDA(cudaMemsetAsync(small_counters, 0, moe::kSmallCounterBytes, s));
  } else {
    MOE_CUDA(moe::launch_prep(pa, s));
  }

  moe::ExpertsArgs ea{};
  ea.wmap = h->wmap;
  ea.stages = h->stages;
  ea.ids = topk_ids;
  ea.plan_codes = pa.plan_codes;
  ea.plan_scales = pa.plan_scales;
  ea.unit_count = pa.unit_count;
  ea.unit_expert = pa.unit_expert;
  ea.unit_rows = pa.unit_rows;
  ea.wide_units = pa.wide_units;
  ea.item_counters = pa.item_counters;
  ea.hidden_flags = pa.hidden_flags;
  ea.partials = reinterpret_cast<float*>(w + offsets[7]);
  ea.hidden = w + offsets[8];
  ea.out = static_cast<uint16_t*>(out_bf16);
  ea.status = h->status_dev;  // read and cleared by moe_sync_status, as for moe_run
  ea.B = batch;
  ea.g = g;
  ea.timeout_ns = h->timeout_ns;
  ea.withhold_unit = -1;
  ea.withhold_image = -1;
  if (small) {
    ea.x = static_cast<const uint16_t*>(x_bf16);
    ea.piece_sums = piece_sums;
    ea.piece_readers = piece_readers;
    ea.small_counters = small_counters;
    ea.seg_cap = small_cap;
    ea.piece_words = small_words;
    ea.parity = 0;
    ea.pair_kept = nullptr;
  }
  MOE_CUDA(moe::launch_experts(ea, h->grid, s, true, h->path, small));
  return MOE_OK;
}

