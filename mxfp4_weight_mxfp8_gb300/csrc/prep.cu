// Kernel 1 (MXFP8 activation plan) and kernel 2 (unit table), launched as one
// grid by moe_run and separately by moe_quantize / moe_group.
//
// Quantizer: page ...cutedsl.moe.experts, mx_block / plan_chunk /
// ExpertsPlanKernel: one E8M0 scale per 32 BF16 values (the smallest E with
// max|x| <= 448 * 2^E), codes e4m3(x * 2^-E). Each thread owns 8 consecutive
// values (one 16-byte load); the four threads of a 32-block combine their
// maxima with two butterfly shuffles, so the result is bit-identical to a
// whole-block maximum.
//
// Grouping: ExpertsKernel.group / ExpertsGroupKernel: per-expert token
// bitmasks (atomic OR), unit counts ceil(n_e / 8), an exclusive scan in
// expert order, and each pair's row = popcount of the lower tokens' bits.
// Experts ascend, rows keep token order, padding is -1. Alongside, the
// table of 16-row units the grid kernel runs for calls of more than 8
// tokens: expert e's units taken two at a time (ceil(units_e / 2) entries,
// in table order), each entry the first unit's index, the expert and
// whether the next unit belongs to it (see kWideFirstMask).
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kPrepThreads = 256;
constexpr int kQuantChunks = 4;  // 256-chunk runs per quantizer block

// One 8-value chunk (a 16-byte load) of the plan, computed in registers: the
// four threads of a 32-block combine their maxima with two butterfly
// shuffles. Stored by store_chunk.
struct PlanChunk {
  uint2 codes;
  int token, c, E;
  bool active;
};

__device__ PlanChunk quantize_chunk(const PrepArgs& a, int chunk) {
  PlanChunk q{};
  const int per_row = a.H / 8;  // 8-value chunks per token
  const int total = a.B * per_row;
  q.active = chunk < total;  // uniform across each 4-lane block (total % 4 == 0)
  q.token = q.active ? chunk / per_row : 0;
  q.c = q.active ? chunk % per_row : 0;
  float v[8];
  float amax = 0.f;
  if (q.active) {
    uint4 w = *reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(q.token) * a.H + q.c * 8);
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(words[i] << 16);
      v[2 * i + 1] = __uint_as_float(words[i] & 0xFFFF0000u);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  if (!q.active) return q;
  q.E = mx_exponent(amax, false);
  const float inv = pow2f(-q.E);
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) lo |= static_cast<uint32_t>(e4m3_code(v[i] * inv)) << (8 * i);
#pragma unroll
  for (int i = 0; i < 4; ++i) hi |= static_cast<uint32_t>(e4m3_code(v[4 + i] * inv)) << (8 * i);
  q.codes = make_uint2(lo, hi);
  return q;
}

__device__ void store_chunk(const PrepArgs& a, const PlanChunk& q) {
  if (!q.active) return;
  *reinterpret_cast<uint2*>(a.plan_codes + static_cast<size_t>(q.token) * a.H + q.c * 8) = q.codes;
  if ((q.c & 3) == 0)
    a.plan_scales[static_cast<size_t>(q.token) * (a.H / kBlock) + q.c / 4] =
        static_cast<uint8_t>(q.E + 127);
}

// Quantizer blocks own kQuantChunks consecutive runs of 256 chunks each: all
// are loaded and quantized first, then (after the previous grid on the
// stream has ended) stored.
__device__ void quantize_role(const PrepArgs& a, int block) {
  PlanChunk q[kQuantChunks];
#pragma unroll
  for (int r = 0; r < kQuantChunks; ++r)
    q[r] = quantize_chunk(a, (block * kQuantChunks + r) * kPrepThreads + threadIdx.x);
  if (!a.early) ptx::grid_dependency_wait();
#pragma unroll
  for (int r = 0; r < kQuantChunks; ++r) store_chunk(a, q[r]);
}

__device__ void group_role(const PrepArgs& a, uint8_t* smem) {
  const int E = a.E, pairs = a.B * kTopK, words = (a.B + 31) / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* masks = reinterpret_cast<uint32_t*>(smem);          // [E][words]
  int32_t* ustart = reinterpret_cast<int32_t*>(masks + E * words);  // [E]
  int32_t* warp_total = ustart + E;                             // [8]
  int32_t* grand = warp_total + 8;                              // [1]

  // Every id this thread handles, loaded in one batch (pair it * 256 + tid).
  constexpr int kIters = MOE_MAX_BATCH * kTopK / kPrepThreads;
  int ev[kIters];
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int p = it * kPrepThreads + tid;
    ev[it] = p < pairs ? a.ids[p] : -1;
  }
  for (int i = tid; i < E * words; i += kPrepThreads) masks[i] = 0;
  __syncthreads();
  // A pair is kept unless its id is out of range or repeats an earlier slot
  // of its token (whichever atomic OR lands first keeps the bit).
  // (Dropped pairs are reported, and the kept flags stored, after the wait
  // below: nothing is written to global memory before it.)
  uint32_t kept_bits = 0;
  bool dropped = false;
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int base = it * kPrepThreads + warp * 32;
    if (it * kPrepThreads >= pairs) break;
    const int p = base + lane;
    bool kept = false;
    if (p < pairs) {
      const int e = ev[it], t = p >> 4;
      if (e >= 0 && e < E) {
        const uint32_t bit = 1u << (t & 31);
        const uint32_t old = atomicOr(&masks[e * words + (t >> 5)], bit);
        kept = !(old & bit);  // else the expert repeats within token t
      }
      dropped |= !kept;
    }
    kept_bits |= static_cast<uint32_t>(kept) << it;
  }
  __syncthreads();

  // Units and pairs of units per expert over a contiguous expert range per
  // thread, then one exclusive scan in expert order of both counts packed
  // into one word (units << 16 | pairs; both stay below 2^15).
  const int span = (E + kPrepThreads - 1) / kPrepThreads;
  const int e0 = tid * span, e1 = min(E, e0 + span);
  int local = 0;
  for (int e = e0; e < e1; ++e) {
    int n = 0;
    for (int w = 0; w < words; ++w) n += __popc(masks[e * words + w]);
    const int un = (n + 7) >> 3;
    local += (un << 16) | ((un + 1) >> 1);
  }
  int incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int other = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += other;
  }
  if (lane == 31) warp_total[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += warp_total[w];
  if (tid == kPrepThreads - 1) *grand = before + incl;
  int start = before + incl - local;
  // The previous grid on the stream may still read the tables written below.
  if (!a.early) ptx::grid_dependency_wait();
  if (dropped) report(a.status, MOE_ERR_DEVICE_IDS);
  if (a.pair_kept != nullptr)
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
      const int p = it * kPrepThreads + tid;
      if (p < pairs) a.pair_kept[p] = (kept_bits >> it) & 1u;
    }
  for (int e = e0; e < e1; ++e) {
    int n = 0;
    for (int w = 0; w < words; ++w) n += __popc(masks[e * words + w]);
    const int un = (n + 7) >> 3, us = start >> 16, ws = start & 0xFFFF;
    ustart[e] = us;
    for (int k = 0; 2 * k < un && ws + k < a.unit_cap; ++k)
      a.wide_units[ws + k] = wide_entry(us + 2 * k, e, 2 * k + 1 < un);
    start += (un << 16) | ((un + 1) >> 1);
  }
  __syncthreads();
  int units = *grand >> 16;
  const int wides = *grand & 0xFFFF;
  if (units > a.unit_cap) {  // cannot happen: units <= 2B + min(E, 16B)
    report(a.status, MOE_ERR_DEVICE_IDS);
    units = 0;
  }
  if (tid == 0) {
    a.unit_count[0] = units;
    a.unit_count[1] = units > 0 ? wides : 0;
  }
  if (units == 0) return;
  // One thread per unit: its expert is the last one whose first unit is at
  // or before it (experts without units share the next one's start). Rows
  // start as padding; the scatter below fills them.
  for (int u = tid; u < units; u += kPrepThreads) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ustart[mid] <= u) lo = mid; else hi = mid - 1;
    }
    a.unit_expert[u] = lo;
    reinterpret_cast<int4*>(a.unit_rows)[u] = make_int4(-1, -1, -1, -1);
  }
  for (int i = tid; i < units * a.P1; i += kPrepThreads) a.item_counters[i] = 0;
  for (int i = tid; i < units * a.KC2; i += kPrepThreads) a.hidden_flags[i] = 0;
  __syncthreads();  // the padding stores precede the row stores
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    if (!((kept_bits >> it) & 1u)) continue;
    const int p = it * kPrepThreads + tid;
    const int e = ev[it], t = p >> 4, w = t >> 5;
    int rank = __popc(masks[e * words + w] & ((1u << (t & 31)) - 1u));
    for (int i = 0; i < w; ++i) rank += __popc(masks[e * words + i]);
    a.unit_rows[(ustart[e] + (rank >> 3)) * kUnitRows + (rank & 7)] = static_cast<int16_t>(p);
  }
}

// Grouping for calls of at most kPrepThreads pairs (16 tokens): thread p owns
// pair p and counts, over all pairs, those of its own expert (before it and
// in total) and the units of all smaller experts. The table is the same
// canonical one (experts ascending, rows in pair order); of two repeated ids
// of a token the lower slot is kept.
__device__ void group_small(const PrepArgs& a, uint8_t* smem) {
  const int pairs = a.B * kTopK, tid = threadIdx.x;
  int32_t* key = reinterpret_cast<int32_t*>(smem);  // [256]: expert of a kept pair, else INT_MAX
  int32_t* nun = key + kPrepThreads;                // [256]: units of the expert, on its first pair
  const int e = tid < pairs ? a.ids[tid] : -1;
  // Lanes 0-15 and 16-31 of a warp hold the 16 slots of one token: a pair is
  // kept when its id is in range and no lower lane of its token has the same
  // id (out-of-range ids get a key of their own).
  const int lane = tid & 31;
  const bool valid = tid < pairs && e >= 0 && e < a.E;
  const unsigned same = __match_any_sync(0xFFFFFFFFu, valid ? 2 * e + ((lane >> 4) & 1) : -1 - lane);
  const bool kept = valid && __ffs(same) - 1 == lane;
  key[tid] = kept ? e : 0x7FFFFFFF;
  __syncthreads();
  // Both loops read four pairs per 16-byte load (pairs is a multiple of 16).
  const int4* key4 = reinterpret_cast<const int4*>(key);
  const int4* nun4 = reinterpret_cast<const int4*>(nun);
  int n = 0, before = 0;
  if (kept)
#pragma unroll 4
    for (int q = 0; q < pairs; q += 4) {
      const int4 k = key4[q >> 2];
      const int s0 = k.x == e, s1 = k.y == e, s2 = k.z == e, s3 = k.w == e;
      n += s0 + s1 + s2 + s3;
      before += (s0 & (q < tid)) + (s1 & (q + 1 < tid)) + (s2 & (q + 2 < tid)) + (s3 & (q + 3 < tid));
    }
  nun[tid] = (kept && before == 0) ? (n + 7) >> 3 : 0;
  __syncthreads();
  // Each expert here has at most 16 pairs: one or two units, one pair of units.
  int units = 0, ubefore = 0, wides = 0, wbefore = 0;
#pragma unroll 4
  for (int q = 0; q < pairs; q += 4) {
    const int4 v = nun4[q >> 2], k = key4[q >> 2];
    units += v.x + v.y + v.z + v.w;
    ubefore += (k.x < e ? v.x : 0) + (k.y < e ? v.y : 0) + (k.z < e ? v.z : 0) + (k.w < e ? v.w : 0);
    wides += (v.x > 0) + (v.y > 0) + (v.z > 0) + (v.w > 0);
    wbefore += (k.x < e && v.x > 0) + (k.y < e && v.y > 0) + (k.z < e && v.z > 0) + (k.w < e && v.w > 0);
  }
  // The previous grid on the stream may still read the tables written below.
  if (!a.early) ptx::grid_dependency_wait();
  if (tid < pairs && !kept) report(a.status, MOE_ERR_DEVICE_IDS);  // out of range or repeated
  if (a.pair_kept != nullptr && tid < pairs) a.pair_kept[tid] = kept ? 1 : 0;
  if (tid == 0) {
    a.unit_count[0] = units;
    a.unit_count[1] = wides;
  }
  if (kept && before == 0) a.wide_units[wbefore] = wide_entry(ubefore, e, n > 8);
  if (kept) {
    const int u = ubefore + (before >> 3), r = before & 7;
    a.unit_rows[u * kUnitRows + r] = static_cast<int16_t>(tid);
    if (r == 0) {  // the unit's first pair: its expert and its padding rows
      a.unit_expert[u] = e;
      for (int rr = min(kUnitRows, n - before); rr < kUnitRows; ++rr) a.unit_rows[u * kUnitRows + rr] = -1;
    }
  }
  for (int i = tid; i < units * a.P1; i += kPrepThreads) a.item_counters[i] = 0;
  for (int i = tid; i < units * a.KC2; i += kPrepThreads) a.hidden_flags[i] = 0;
}

// Chained to the previous launch on the stream (programmatic dependent
// launch): every role reads ids and x and does its work in registers and
// shared memory first, and waits for the previous grid to end only before
// its first global write, so that work overlaps the previous experts
// kernel's tail. ids and x themselves are read at once (see moe_run).
__global__ void __launch_bounds__(kPrepThreads, 6) prep_kernel(const PrepArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  // Let the call's experts kernel start its prologue; it waits for this
  // grid's end (or, started early, for the tables' flag) before reading
  // anything written here.
  if (a.chained) ptx::grid_launch_dependents();
  // The grouping block is block 0, dispatched first: it has the longest run.
  const int group_blocks = (a.roles & kPrepGroup) ? 1 : 0;
  if (group_blocks && blockIdx.x == 0) {
    if (a.B * kTopK <= kPrepThreads)
      group_small(a, smem);
    else
      group_role(a, smem);
  } else if (a.roles & kPrepQuantize) {
    quantize_role(a, blockIdx.x - group_blocks);
  }
  if (a.early) {
    // Every block's writes are out before the last one raises the flag. The
    // grid still ends only after the previous grid has (its last block waits
    // for it; the others leave at once, freeing their SMs for the experts
    // kernel), so that the experts kernel's wait for this grid covers that
    // one too.
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(a.arrive, 1u) == gridDim.x - 1) {
        *a.arrive = 0u;
        __threadfence();
        ptx::store_release_gpu(a.ready, a.seq);
      }
    }
    if (blockIdx.x == gridDim.x - 1) ptx::grid_dependency_wait();
  }
}

}  // namespace

int prep_group_smem_bytes(int experts) {
  const int words = (MOE_MAX_BATCH + 31) / 32;
  const int general = experts * words * 4 + experts * 4 + 9 * 4;
  const int small = 2 * kPrepThreads * 4;  // group_small's two arrays
  return general > small ? general : small;
}

int prep_quant_blocks(int batch, int hidden) {
  const int chunks = batch * (hidden / 8);
  return (chunks + kPrepThreads * kQuantChunks - 1) / (kPrepThreads * kQuantChunks);
}

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t stream) {
  int blocks = 0;
  if (a.roles & kPrepQuantize) blocks += a.quant_blocks;
  if (a.roles & kPrepGroup) blocks += 1;
  if (blocks == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kPrepThreads);
  cfg.dynamicSmemBytes = (a.roles & kPrepGroup) ? prep_group_smem_bytes(a.E) : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prep_kernel, a);
}

}  // namespace moe
