// Device-side building blocks shared by the experts kernels (the persistent
// grid kernel, its cluster variant and the small-batch kernel): the
// shared-memory carve-up, the per-call work split, bounded mbarrier waits and
// the epilogue's abort agreement, the launch clock and phase stamps, and the
// FC1 / FC2 work cursors. Each translation unit that includes it gets its own
// copy (internal linkage).
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int S = kRingStages;
constexpr int NACC = kAccSets;
constexpr int kHalvesFrom = 256;  // more units than this: split them into halves A and B
constexpr int kRowCache = 16;    // unit rows the epilogue keeps in shared memory
constexpr int kAgreeSlots = 2 * NACC;  // epilogue decisions in flight after an abort
static_assert(kAgreeSlots >= 2 * Rows<16>::kSets, "agreement slots for every unit size");
constexpr uint32_t kWaitHintNs = 20000;  // longest suspension of one mbarrier wait step
// The grid kernel keeps every unit's expert (R = 8: unit_expert; R = 16: the
// pair-table entry) in shared memory: at most 2B + min(E, 16B) units, B <= 8
// and B <= 256 (E <= 1024).
constexpr int kUnitCache8 = 2 * 8 + 16 * 8;
constexpr int kUnitCache16 = 2 * MOE_MAX_BATCH + MOE_MAX_EXPERTS;

// Shared-memory carve-up. The swizzled operand images (weights, activation
// and hidden codes) start on 1024-byte boundaries, every other region on a
// 16-byte boundary (mbarriers need 8, int4 metadata and uint4 copies 16).
// Units of `rows` rows (8, or 16 in the grid kernel's larger calls) set the
// ring depth, the accumulator sets and the image sizes (Rows<R>). The grid
// kernel (`grid`) packs the per-slot activation scale atoms R x 16 bytes
// apart: only rows 0..R-1 of an atom are written and used (the 32-row copy
// of slot s reads slot s + 1's rows into TMEM lanes that an N = R MMA never
// reads), and only the last atom is a full 512 bytes.
struct Layout {
  int w, act, asf, hcodes, out, bsf, hsf, table, bars, meta, misc, rows, agree, units, bytes;
  __host__ __device__ static int up(int o, int a) { return (o + a - 1) / a * a; }
  int bsf_stride;
  __host__ __device__ explicit Layout(int kc2, int unit_rows = 8, bool grid = false) {
    const int slots = unit_rows == 8 ? Rows<8>::kSlots : Rows<16>::kSlots;
    const int sets = unit_rows == 8 ? Rows<8>::kSets : Rows<16>::kSets;
    const int image = unit_rows * kChunkK;
    int o = 0;
    w = o;                 o += slots * kStageSmemWeights;
    act = o = up(o, 1024); o += slots * image;
    hcodes = o = up(o, 1024); o += 2 * kc2 * image;
    asf = o = up(o, 16);   o += slots * 2 * kScaleAtomBytes;
    out = o = up(o, 16);   o += unit_rows * 2 * kTileM * 2;
    bsf_stride = grid ? unit_rows * 16 : kScaleAtomBytes;
    bsf = o = up(o, 16);   o += (slots - 1) * bsf_stride + kScaleAtomBytes;
    hsf = o = up(o, 16);   o += 2 * kc2 * kScaleAtomBytes;
    table = o = up(o, 16); o += 2 * (kMaxGrid + 1) * 4;
    // full, empty (+ the grid kernel's scaled) per slot, accfull/accempty per
    // set, hfull/hempty, drained per issuer (+ per copier).
    bars = o = up(o, 16);  o += ((grid ? 3 : 2) * slots + 2 * sets + 4 + kMmaWarps + (grid ? kCopiers : 0)) * 8;
    meta = o = up(o, 16);  o += sets * 16;
    misc = o = up(o, 16);  o += 16;
    rows = o = up(o, 16);  o += kRowCache * ((grid ? 12 : 8) + unit_rows * 2);
    agree = o = up(o, 16); o += kAgreeSlots * 4;
    units = o = up(o, 16); o += grid ? (unit_rows == 8 ? kUnitCache8 : kUnitCache16) * 4 : 0;
    bytes = o + 1024;  // slack for aligning the dynamic shared-memory base to 1024
  }
  __host__ __device__ bool aligned() const {
    return w % 1024 == 0 && act % 1024 == 0 && hcodes % 1024 == 0 && asf % 16 == 0 &&
           out % 16 == 0 && bsf % 16 == 0 && hsf % 16 == 0 && table % 16 == 0 && bars % 16 == 0 &&
           meta % 16 == 0 && misc % 16 == 0 && rows % 16 == 0 && agree % 16 == 0 && units % 16 == 0;
  }
};

// Per-call split of the work over the grid: FC1 stages and FC2 jobs are each
// cut evenly over the CTAs. A unit's FC2 waits for its hidden vector, which is
// complete only when the FC1 ranges holding its items are done, so the FC1
// ranges are kept equal rather than evening out FC1 + FC2 stages per CTA.
// Every CTA computes the same table.
struct Split {
  int T1, J, G, skew;
  __host__ __device__ Split(int units, const Geometry& g, int grid, int skewed = 0) {
    T1 = units * g.P1 * g.KC1;
    J = units * g.NQ;
    G = grid;
    skew = skewed;
  }
  // 32-bit products: T1 <= 2M stages and c <= 256 for every supported layer.
  __host__ __device__ int fc2_begin(int c) const {
    const uint32_t cu = static_cast<uint32_t>(c);
    return static_cast<int>(cu * static_cast<uint32_t>(J) / static_cast<uint32_t>(G));
  }
  // The CTA holding FC2 job j: the largest c < G with fc2_begin(c) <= j.
  __host__ __device__ int job_owner(int j) const {
    const int c = static_cast<int>((static_cast<uint32_t>(j + 1) * static_cast<uint32_t>(G) - 1u) /
                                   static_cast<uint32_t>(J));
    return c < G - 1 ? c : G - 1;
  }
  // Even FC1 ranges, or (skewed) ranges that favour the low CTAs: CTA c's
  // range then starts at T1 * x * (1 + (1 - x) / 4), x = c / G. A call that
  // starts while the previous one still runs gets its CTAs in block order as
  // the previous call's leave, so the ones that start first take up to a
  // quarter more stages and all finish FC1 closer together.
  __host__ __device__ int fc1_begin(int c) const {
    if (c >= G) return T1;
    const uint64_t cu = static_cast<uint64_t>(c), g = static_cast<uint64_t>(G);
    if (!skew) return static_cast<int>(cu * static_cast<uint64_t>(T1) / g);
    return static_cast<int>(static_cast<uint64_t>(T1) * cu * (5ull * g - cu) / (4ull * g * g));
  }
};

struct Ctx {
  const ExpertsArgs* a;
  volatile uint32_t* abort_flag;
};

// Bounded mbarrier wait: false after the time limit (recording the error)
// or once another role of this CTA has given up.
__device__ bool wait_bar(const Ctx& cx, uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t start = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_wait_hint(bar, parity, kWaitHintNs)) return true;
    if ((i & 7u) == 0) {
      if (*cx.abort_flag) return false;
      if (global_timer_ns() - start > cx.a->timeout_ns) {
        *cx.abort_flag = 1;
        report(cx.a->status, MOE_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

// wait_bar for barriers that other CTAs of the cluster arrive on.
__device__ bool wait_bar_cluster(const Ctx& cx, uint64_t* bar, uint32_t parity) {
  if (mbar_test_cluster(bar, parity)) return true;
  const uint64_t start = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test_cluster(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*cx.abort_flag) return false;
      if (global_timer_ns() - start > cx.a->timeout_ns) {
        *cx.abort_flag = 1;
        report(cx.a->status, MOE_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Bounded wait on a completion that is bound to come (this thread's own
// tensor-core work, or a barrier another thread has seen complete), taken
// after a failure as well: the abort flag does not end it.
__device__ void wait_own(const Ctx& cx, uint64_t* bar, uint32_t parity) {
  const uint64_t start = global_timer_ns();
  for (uint32_t i = 1; !mbar_test(bar, parity); ++i) {
    if ((i & 63u) == 0 && global_timer_ns() - start > cx.a->timeout_ns) {
      report(cx.a->status, MOE_ERR_DEVICE_TIMEOUT);
      return;
    }
  }
}

// The epilogue threads' common decision on accumulator k (true: process it).
// A thread that saw the barrier complete and then the abort flag still clear
// goes on: the barrier completed before any abort. Any other thread calls
// this: it tests the barrier once more and proposes to go on if it has
// completed, to stop if not; the first proposal for k, kept by
// compare-and-swap, decides for every such thread. The two kinds agree, as a
// proposal to stop shows that the barrier had not completed when the abort
// came. So no epilogue warp goes on into a named barrier that another has
// left. A thread runs at most NACC accumulators ahead of another, so
// 2 * NACC slots keep the decisions in flight apart.
__device__ __noinline__ bool epilogue_agree(const Ctx& cx, uint64_t* bar, uint32_t parity, int k, int* agree) {
  const int proposal = (k << 2) | (mbar_test(bar, parity) ? 1 : 2);
  int* slot = agree + (k & (kAgreeSlots - 1));
  int v = *reinterpret_cast<volatile int*>(slot);
  while ((v >> 2) != k) {
    const int w = atomicCAS(slot, v, proposal);
    v = w == v ? proposal : w;
  }
  if ((v & 3) != 1) return false;
  wait_own(cx, bar, parity);  // completed already: some thread saw it
  return true;
}

// After a failed wait nobody waits for the copies still in flight into (or
// out of) this CTA's shared memory: give them 50 us to land before it exits.
__device__ void settle_copies() {
  const uint64_t start = global_timer_ns();
  while (global_timer_ns() - start < 50000) __nanosleep(1000);
}

// Release increment (no result): the caller's earlier stores, and those of
// the threads it synchronized with, are visible to whoever acquires the count.
__device__ __forceinline__ void red_release_add_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Launch clock (moe_debug_kernel_span): CTA c stores its start and end times
// (%globaltimer) into words 2c and 2c + 1; plain stores, so the clock costs
// the launch nothing measurable. The host reduces them to the launch's span.
__device__ __forceinline__ void span_enter(uint64_t* span) {
  if (span != nullptr && blockIdx.x < kMaxSpanCtas) span[2 * blockIdx.x] = global_timer_ns();
}

__device__ __forceinline__ void span_leave(uint64_t* span) {
  if (span != nullptr && blockIdx.x < kMaxSpanCtas) span[2 * blockIdx.x + 1] = global_timer_ns();
}

// Phase stamps for timing studies, compiled in only with -DMOE_TRACE: slot k
// of this CTA's 32-word record gets the time the CTA passed point k.
#ifdef MOE_TRACE
#define MOE_STAMP(k)                                                                        \
  do {                                                                                      \
    if (a.trace != nullptr) a.trace[static_cast<size_t>(blockIdx.x) * 32 + (k)] = global_timer_ns(); \
  } while (0)
#define MOE_STAMP_VALUE(k, v)                                                              \
  do {                                                                                     \
    if (a.trace != nullptr) a.trace[static_cast<size_t>(blockIdx.x) * 32 + (k)] = (v);     \
  } while (0)
#else
#define MOE_STAMP(k) \
  do {               \
  } while (0)
#define MOE_STAMP_VALUE(k, v) \
  do {                        \
  } while (0)
#endif

// The largest |v| over the 32 lanes of the warp, in one warp reduction: for
// non-negative floats (finite or infinite) the order of the bit patterns as
// unsigned integers is the order of the values.
__device__ __forceinline__ float warp_amax(float v) {
  return __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(v))));
}

// One output row segment of a warp: lane l holds the value of column l of
// 32 consecutive BF16 outputs at `dst` (16-byte aligned). Adjacent lanes pair
// their values into 32-bit words, and lane 8j gathers the words of lanes 8j,
// 8j + 2, 8j + 4, 8j + 6 and stores columns 8j .. 8j + 7 as one 16-byte store.
// Every lane of the warp must call it.
__device__ __forceinline__ void store_row32_bf16(uint16_t* dst, float v, int lane) {
  const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  const uint32_t pair = b | (__shfl_down_sync(0xFFFFFFFFu, b, 1) << 16);
  const uint32_t w1 = __shfl_down_sync(0xFFFFFFFFu, pair, 2);
  const uint32_t w2 = __shfl_down_sync(0xFFFFFFFFu, pair, 4);
  const uint32_t w3 = __shfl_down_sync(0xFFFFFFFFu, pair, 6);
  if ((lane & 7) == 0) *reinterpret_cast<uint4*>(dst + lane) = make_uint4(pair, w1, w2, w3);
}

__device__ __forceinline__ float silu_times(float gate, float up) {
  return gate / (1.0f + expf(-gate)) * up;
}

__device__ __forceinline__ uint64_t desc_sw128(const void* p) {
  return smem_desc(smem_addr(p), 16, 1024, 2);
}
__device__ __forceinline__ uint64_t desc_scales(const void* p) {
  return smem_desc(smem_addr(p), 128, 128, 0);
}

// FC1 stage cursor: stage s = (item * KC1 + c), item = u * P1 + p.
struct Fc1Cursor {
  int s, item, c, u, p;
  __device__ Fc1Cursor(int s0, const Geometry& g) : s(s0) {
    item = s0 / g.KC1;
    c = s0 - item * g.KC1;
    u = item / g.P1;
    p = item - u * g.P1;
  }
  __device__ void next(const Geometry& g) {
    ++s;
    if (++c == g.KC1) {
      c = 0;
      ++item;
      if (++p == g.P1) {
        p = 0;
        ++u;
      }
    }
  }
};

// FC2 job cursor: job j = u * NQ + q.
struct Fc2Cursor {
  int j, u, q;
  __device__ Fc2Cursor(int j0, const Geometry& g) : j(j0) {
    u = j0 / g.NQ;
    q = j0 - u * g.NQ;
  }
  __device__ void next(const Geometry& g) {
    ++j;
    if (++q == g.NQ) {
      q = 0;
      ++u;
    }
  }
};

}  // namespace
}  // namespace moe
