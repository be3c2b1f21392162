// Kernel 3 (+4): the persistent experts kernel with its BF16 output epilogue.
//
// Pages: ...cutedsl.moe.experts (ExpertsKernel: the TMA producer warp, the
// block-scaled FC1/FC2 tcgen05 stages, store_hidden, the hidden exchange,
// fc2 output rows) and ...cutedsl.moe.experts_runtime (PersistentExperts:
// one co-resident persistent grid, per-call workspace).
//
// One CTA per SM, 10 warps:
//   warp 0     TMA producer: one 17 KB stage per ring slot (two 128-row e2m1
//              tiles x 128 K, expanded to 32 KB of 8-bit slots in shared
//              memory with the 128-byte swizzle, plus 1 KB of pre-tiled scales)
//   warps 1-4  MMA issuers. Issuer i owns tile i / 2 and K-steps
//              2 (i % 2), 2 (i % 2) + 1 of every stage: it copies its scale
//              atoms into TMEM and issues tcgen05.mma kind::mxf8f6f4.block_scale
//              (M = 128 weight rows, N = 8 unit rows, K = 32) into its own
//              accumulator. One thread issues an MMA about every hundred
//              cycles, so four issuers keep up with HBM.
//   warp 5     FC1: cp.async gather of each stage's 8 MXFP8 activation rows;
//              FC2: bounded wait for each unit's hidden vector, then a copy of
//              its image into shared memory
//   warps 6-9  epilogue: FC1 -> split-K reduction, SiLU(gate) * up, MXFP8
//              hidden requant, publish; FC2 -> BF16 rows with 16-byte stores
//
// Work split: FC1 stages (unit, tile pair, K chunk) and FC2 jobs (unit, 256
// output rows) are each cut evenly into contiguous per-CTA ranges, and every
// CTA runs its FC1 range, then its FC2 range. Above 256 units the
// units are cut into two halves, A and B, run as FC1(A), FC1(B), FC2(A),
// FC2(B): half A's hidden vectors are reduced and published while half B's
// FC1 weights stream.
// An FC1 item split across CTAs is reduced by the CTA holding its first
// stage: the others store FP32 partial sums and release-increment a counter
// that the owner acquires; a fixed CTA order keeps the sum deterministic.
// Every wait is bounded by a time limit.
//
// Calls of one or two tokens run on cluster_kernel (below) instead: one
// thread-block cluster per unit, the same roles and stages, and the two
// hand-offs through distributed shared memory.
#include "pipeline.cuh"

namespace moe {
namespace {

using namespace ptx;

// Unit u of a launch with R-row units: the table's unit u (R = 8), or the
// pair-table entry u (R = 16; see kWideFirstMask). `xc` is the shared-memory
// copy of unit_expert (R = 8) or of the pair table (R = 16).
template <int R>
__device__ __forceinline__ int unit_first_of(const uint32_t* xc, int u) {
  if constexpr (R == 8) return u;
  else return static_cast<int>(xc[u] & kWideFirstMask);
}

template <int R>
__device__ __forceinline__ int unit_expert_of(const uint32_t* xc, int u) {
  if constexpr (R == 8) return static_cast<int>(xc[u]);
  else return static_cast<int>((xc[u] >> 20) & 0x3FFu);
}

// Rows of table unit tu: its pairs, then -1 padding (one 16-byte load).
__device__ __forceinline__ int table_unit_valid(const ExpertsArgs& a, int tu) {
  const int4 r4 = __ldcg(reinterpret_cast<const int4*>(a.unit_rows) + tu);
  const uint32_t w4[4] = {static_cast<uint32_t>(r4.x), static_cast<uint32_t>(r4.y),
                          static_cast<uint32_t>(r4.z), static_cast<uint32_t>(r4.w)};
  int v = 0;
#pragma unroll
  for (int r = 0; r < kUnitRows; ++r) v += static_cast<int16_t>(w4[r >> 1] >> (16 * (r & 1))) >= 0;
  return v;
}

// Row r of unit u: a pair index (token * 16 + slot) or -1 (padding). A
// pair's rows 8-15 are the second table unit's, which follows the first.
template <int R>
__device__ __forceinline__ int unit_row_of(const ExpertsArgs& a, const uint32_t* xc, int u, int r) {
  if constexpr (R == 8) {
    return a.unit_rows[u * kUnitRows + r];
  } else {
    const uint32_t w = xc[u];
    const int first = static_cast<int>(w & kWideFirstMask);
    return (r < kUnitRows || (w >> 31)) ? a.unit_rows[first * kUnitRows + r] : -1;
  }
}

template <int R>
__global__ void __launch_bounds__(kGridThreads, 1) experts_kernel(const __grid_constant__ ExpertsArgs a) {
  // R rows per unit: the table's units (R = 8) or pairs of them (R = 16).
  using RT = Rows<R>;
  constexpr int S = RT::kSlots;
  constexpr int NACC = RT::kSets;
  constexpr int kImage = RT::kImage;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const Geometry& g = a.g;
  const Layout L(g.KC2, R, true);
  uint8_t* W = sm + L.w;
  uint8_t* ACT = sm + L.act;
  uint8_t* ASF = sm + L.asf;
  uint8_t* HC = sm + L.hcodes;
  uint16_t* OUT = reinterpret_cast<uint16_t*>(sm + L.out);
  uint8_t* BSF = sm + L.bsf;
  uint8_t* HSF = sm + L.hsf;
  int* start = reinterpret_cast<int*>(sm + L.table);  // FC1 range starts, [2 halves][G + 1]
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + S;
  uint64_t* accfull = empty + S;
  uint64_t* accempty = accfull + NACC;
  uint64_t* hfull = accempty + NACC;
  uint64_t* hempty = hfull + 2;
  uint64_t* drained = hempty + 2;  // [issuer, then copier]: its tensor-core work has finished
  uint64_t* scaled = drained + kMmaWarps + kCopiers;  // [slot]: the stage's scale atoms are in TMEM
  int* agree = reinterpret_cast<int*>(sm + L.agree);
  int4* meta = reinterpret_cast<int4*>(sm + L.meta);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + L.misc);  // tmem base, abort, last flag

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  Ctx cx{&a, reinterpret_cast<volatile uint32_t*>(&misc[1])};

  if (tid == 0) {
    span_enter(a.span);
    MOE_STAMP(0);
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1 + 32);       // producer (with bytes) + 32 gather lanes or a stand-in
      mbar_init(&empty[s], kMmaWarps);   // one commit per issuer
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&accfull[i], kMmaWarps + 1);  // issuer commits + the metadata arrival
      mbar_init(&accempty[i], 4);             // one per epilogue warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&hfull[b], 1);
      mbar_init(&hempty[b], kMmaWarps);
    }
    misc[1] = 0;
    misc[2] = 0;
    fence_mbar_init();
    prefetch_tensormap(&a.wmap);
  } else if (warp == kMmaWarp0 + 1 && lane == 0) {
    for (int i = 0; i < kMmaWarps + kCopiers; ++i) mbar_init(&drained[i], 1);
    for (int s = 0; s < S; ++s) mbar_init(&scaled[s], kCopiers);  // one commit per copier
    for (int i = 0; i < kAgreeSlots; ++i) agree[i] = -1;
    fence_mbar_init();
  }
  for (int i = tid; i < ((S - 1) * L.bsf_stride + kScaleAtomBytes) / 16; i += kGridThreads)
    reinterpret_cast<uint4*>(BSF)[i] = make_uint4(0, 0, 0, 0);
  if (warp == kMmaWarp0) {
    tmem_alloc(&misc[0], kTmemColumns);
    tmem_relinquish();
  }

  // The plan, unit table and cleared counters of the preceding prep grid.
  // Every unit's expert goes to shared memory in the same round trip as the
  // unit count (entries past the count are never used).
  if (a.early) {
    // The prep grid raised `ready` to this call's number once its writes
    // were out, without waiting for the previous experts grid (another
    // handle's, still running on the other SMs).
    if (tid == 0) {
      const uint64_t t_start = global_timer_ns();
      for (uint32_t i = 0; load_acquire_gpu(a.ready) != a.seq; ++i) {
        __nanosleep(64);
        if ((i & 15u) == 15u && global_timer_ns() - t_start > a.timeout_ns) {
          report(a.status, MOE_ERR_DEVICE_TIMEOUT);
          misc[1] = 1u;
          break;
        }
      }
      if (misc[1] == 0u && atomicAdd(a.passed, 1u) == static_cast<uint32_t>(G) - 1u) {
        *a.passed = 0u;
        *reinterpret_cast<volatile uint32_t*>(a.ready) = 0u;
      }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (misc[1] != 0u) {
      // No tables: end without reading them, after the previous grid.
      if (warp == kMmaWarp0) tmem_dealloc(misc[0], kTmemColumns);
      grid_dependency_wait();
      if (tid == 0) span_leave(a.span);
      return;
    }
  } else {
    grid_dependency_wait();
    // The next call's prep grid may start now: the grid before this one has
    // ended, and it writes nothing before it has waited for this grid to end.
    if (tid == 0) grid_launch_dependents();
  }
  uint32_t* xc = reinterpret_cast<uint32_t*>(sm + L.units);
  {
    const int cap = min(2 * a.B + min(g.E, kTopK * a.B), R == 8 ? kUnitCache8 : kUnitCache16);
    const uint32_t* src = R == 8 ? reinterpret_cast<const uint32_t*>(a.unit_expert) : a.wide_units;
    for (int i = tid; i < cap; i += kGridThreads) xc[i] = src[i];
  }
  const int units = a.unit_count[R == 8 ? 0 : 1];
  if (tid == 0) MOE_STAMP(3);
  // Half A = units [0, units_a). Small calls keep one half: their chain of
  // reductions is latency-bound and more pieces per item only lengthen it.
  const int units_a = units > kHalvesFrom ? (units + 1) / 2 : units;
  const Split half[2] = {Split(units_a, g, G, a.skew), Split(units - units_a, g, G, a.skew)};
  const int stage_base[2] = {0, units_a * g.P1 * g.KC1};
  const int job_base[2] = {0, units_a * g.NQ};
  const int items_a = units_a * g.P1;
  for (int c = tid; c <= G; c += kGridThreads) {
    start[c] = half[0].fc1_begin(c);
    start[G + 1 + c] = stage_base[1] + half[1].fc1_begin(c);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (tid == 0) MOE_STAMP(16);
  const uint32_t tmem = misc[0];
  int f0[2], f1[2], j0[2], j1[2];
  for (int h = 0; h < 2; ++h) {
    f0[h] = start[h * (G + 1) + cta];
    f1[h] = start[h * (G + 1) + cta + 1];
    j0[h] = job_base[h] + half[h].fc2_begin(cta);
    j1[h] = job_base[h] + half[h].fc2_begin(cta + 1);
  }
  const int fc1_stages = g.P1 * g.KC1;  // FC2 stages follow the FC1 stages of an expert

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t policy = policy_evict_first();
      int n = 0, slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      auto issue = [&](int stage, bool stand_in) {
        if (n >= S && !wait_bar(cx, &empty[slot], phase ^ 1)) return false;
        mbar_arrive_expect_tx(&full[slot], kStageWeightBytes + 2 * kScaleAtomBytes);
        if (stand_in) mbar_arrive_count(&full[slot], 32);
        tma_load_3d(W + slot * kStageSmemWeights, &a.wmap, 0, 0, stage, &full[slot], policy);
        bulk_load(ASF + slot * 2 * kScaleAtomBytes,
                  a.stages + static_cast<size_t>(stage) * kStageBytes + kStageWeightBytes,
                  2 * kScaleAtomBytes, &full[slot], policy);
        if (n == 0) MOE_STAMP(1);
        MOE_STAMP(2);
        ++n;
        if (++slot == S) {
          slot = 0;
          phase ^= 1;
        }
        return true;
      };
      int cu = -1, e = 0;
      for (int h = 0; h < 2; ++h)
        for (Fc1Cursor cur(f0[h], g); cur.s < f1[h] && ok; cur.next(g)) {
          if (cur.u != cu) { e = unit_expert_of<R>(xc, cur.u); cu = cur.u; }
          ok = issue(e * g.SPE + cur.p * g.KC1 + cur.c, false);
        }
      cu = -1;
      for (int h = 0; h < 2; ++h)
        for (Fc2Cursor cur(j0[h], g); cur.j < j1[h] && ok; cur.next(g)) {
          if (cur.u != cu) { e = unit_expert_of<R>(xc, cur.u); cu = cur.u; }
          const int base = e * g.SPE + fc1_stages + cur.q * g.KC2;
          for (int c = 0; c < g.KC2 && ok; ++c) ok = issue(base + c, true);
        }
      MOE_STAMP_VALUE(15, static_cast<uint64_t>(n));
      // Drain: every issued stage consumed and released before exit.
      if (ok)
        for (int k = (n > S ? n - S : 0); k < n && ok; ++k) ok = wait_bar(cx, &empty[k % S], (k / S) & 1);
      if (!ok) settle_copies();
    }
  } else if (warp >= kMmaWarp0 && warp < kMmaWarp0 + kMmaWarps) {
    // --------------------------------------------------------- MMA issuers
    if (lane == 0) {
      const int issuer = warp - kMmaWarp0, t = issuer >> 1, k0 = 2 * (issuer & 1);
      const bool lead = issuer == 0;  // writes the accumulator metadata
      const uint32_t hsf_cols = tmem + RT::kHiddenScaleBase + issuer * kHiddenScaleColumns;
      int n = 0, slot = 0, k = 0, ordinal = -1, cu = -1, hb = 0, first_c = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool fc2_seen = false;
      (void)fc2_seen;
      auto acquire = [&](int set) {
        return k < NACC || wait_bar(cx, &accempty[set], ((k / NACC) - 1) & 1);
      };
      auto advance = [&]() {
        ++n;
        if (++slot == S) {
          slot = 0;
          phase ^= 1;
        }
      };
      for (int hf = 0; hf < 2; ++hf)
      for (Fc1Cursor cur(f0[hf], g); cur.s < f1[hf] && ok; cur.next(g)) {
        const bool first = (cur.s == f0[hf]) || (cur.c == 0);
        const bool last = (cur.s == f1[hf] - 1) || (cur.c == g.KC1 - 1);
        const int set = k % NACC;
        if (first) {
          if (!(ok = acquire(set))) break;
          first_c = cur.c;
        }
        // The scale barrier completes only after the copiers have seen the
        // slot's full barrier (weights and activations landed): one wait.
        if (!(ok = wait_bar(cx, &scaled[slot], phase))) break;
        if (lead && n == 0) MOE_STAMP(4);
        fence_proxy_async_shared();  // the gathered activations were cp.async (generic) writes
        tc_fence_after_sync();
        // The slot's scale atoms: tile 0's weights, tile 1's, the activations.
        const uint32_t sf = tmem + RT::kScaleBase + slot * kSlotScaleColumns;
        const uint64_t dw = desc_sw128(W + slot * kStageSmemWeights + t * (kStageSmemWeights / 2) + k0 * 32);
        const uint64_t dx = desc_sw128(ACT + slot * kImage + k0 * 32);
        const uint32_t d = tmem + set * RT::kSetColumns + issuer * R;
        // Descriptor start addresses count 16-byte units: +2 is the next K-step.
        tc_mma_mxf8f6f4(d, dw, dx, mma_idesc(k0, R), sf + 4 * t, sf + 8, first ? 0u : 1u);
        tc_mma_mxf8f6f4(d, dw + 2, dx + 2, mma_idesc(k0 + 1, R), sf + 4 * t, sf + 8, 1u);
        if (lead) MOE_STAMP(5);
        tc_commit(&empty[slot]);
        advance();
        if (last) {
          // (FC1, item, piece starts the item's K range, piece ends it)
          if (lead) meta[set] = make_int4(0, cur.item, first_c == 0, cur.c == g.KC1 - 1);
          tc_commit(&accfull[set]);
          if (lead) mbar_arrive(&accfull[set]);
          ++k;
        }
      }
      for (int hf = 0; hf < 2; ++hf)
      for (Fc2Cursor cur(j0[hf], g); cur.j < j1[hf] && ok; cur.next(g)) {
        if (cur.u != cu) {
          if (cu >= 0) tc_commit(&hempty[hb]);
          ++ordinal;
          hb = ordinal & 1;
          if (!(ok = wait_bar(cx, &hfull[hb], (ordinal >> 1) & 1))) break;
          tc_fence_after_sync();
          // The unit's hidden scale atoms, once for all its jobs.
          for (int c = 0; c < g.KC2; ++c)
            tc_copy_scales(hsf_cols + hb * 16 + c * 4, desc_scales(HSF + (hb * g.KC2 + c) * kScaleAtomBytes));
          cu = cur.u;
        }
        const int set = k % NACC;
        if (!(ok = acquire(set))) break;
        bool started = false;
        for (int c = 0; c < g.KC2 && ok; ++c) {
          if (!(ok = wait_bar(cx, &scaled[slot], phase))) break;  // implies full (see FC1)
          if (lead && !fc2_seen) {
            MOE_STAMP(10);
            fc2_seen = true;
          }
          tc_fence_after_sync();
          // K-steps of this chunk: 4, or fewer in the last chunk when I % 128 != 0.
          const int ksteps = c + 1 < g.KC2 ? 4 : (g.I - c * kChunkK) / kBlock;
          if (k0 < ksteps) {
            const uint32_t sf = tmem + RT::kScaleBase + slot * kSlotScaleColumns + 4 * t;
            const int hc = hb * g.KC2 + c;
            const uint32_t sfh = hsf_cols + hb * 16 + c * 4;
            const uint64_t dw = desc_sw128(W + slot * kStageSmemWeights + t * (kStageSmemWeights / 2) + k0 * 32);
            const uint64_t dh = desc_sw128(HC + hc * kImage + k0 * 32);
            const uint32_t d = tmem + set * RT::kSetColumns + issuer * R;
            // Descriptor start addresses count 16-byte units: +2 is the next K-step.
            tc_mma_mxf8f6f4(d, dw, dh, mma_idesc(k0, R), sf, sfh, started ? 1u : 0u);
            if (k0 + 1 < ksteps)
              tc_mma_mxf8f6f4(d, dw + 2, dh + 2, mma_idesc(k0 + 1, R), sf, sfh, 1u);
            started = true;
          }
          if (lead) MOE_STAMP(11);
          tc_commit(&empty[slot]);
          advance();
        }
        if (!ok) break;
        if (lead) meta[set] = make_int4(1, cur.j, 0, 0);
        tc_commit(&accfull[set]);
        if (lead) mbar_arrive(&accfull[set]);
        ++k;
      }
      // End marker for the epilogue, only when every wait of this CTA has
      // succeeded: after a failure the issuers may have stopped at different
      // jobs, and a full-count arrival could overrun a barrier that another
      // issuer's commit has reached. The epilogue then ends on the abort flag.
      if (lead && ok && !*cx.abort_flag) {
        const int set = k % NACC;
        if (k < NACC || wait_bar(cx, &accempty[set], ((k / NACC) - 1) & 1)) {
          meta[set] = make_int4(2, 0, 0, 0);
          mbar_arrive_count(&accfull[set], kMmaWarps + 1);
        }
      }
      // The tensor memory is freed only after every MMA and scale copy of
      // this thread has finished (after a failure nobody else waits on them).
      tc_commit(&drained[issuer]);
      wait_own(cx, &drained[issuer], 0);
    }
  } else if (warp >= kCopierWarp0) {
    // ----------------------------------------------------------- scale copies
    // Copier 0 copies tile 0's weight scales and (FC1) the activation scales
    // of every stage, copier 1 tile 1's, into the slot's TMEM columns, and
    // each commits to the slot's `scaled` barrier, which the issuers wait on
    // in place of the full barrier: the copiers wait on that one first, so a
    // completed `scaled` phase is ordered after the stage's data landed.
    // The slot is refilled only after the issuers' MMAs (which waited on
    // these copies) are done, so the columns are free again by then.
    if (lane == 0) {
      const int c = warp - kCopierWarp0;
      int slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      auto copy = [&](bool activations) {
        if (!(ok = wait_bar(cx, &full[slot], phase))) return;
        fence_proxy_async_shared();  // the activation scales were cp.async (generic) writes
        tc_fence_after_sync();
        const uint32_t sf = tmem + RT::kScaleBase + slot * kSlotScaleColumns;
        tc_copy_scales(sf + 4 * c, desc_scales(ASF + slot * 2 * kScaleAtomBytes + c * kScaleAtomBytes));
        if (activations && c == 0) tc_copy_scales(sf + 8, desc_scales(BSF + slot * L.bsf_stride));
        tc_commit(&scaled[slot]);
        if (++slot == S) {
          slot = 0;
          phase ^= 1;
        }
      };
      for (int hf = 0; hf < 2; ++hf)
        for (Fc1Cursor cur(f0[hf], g); cur.s < f1[hf] && ok; cur.next(g)) copy(true);
      for (int hf = 0; hf < 2; ++hf)
        for (Fc2Cursor cur(j0[hf], g); cur.j < j1[hf] && ok; cur.next(g))
          for (int cc = 0; cc < g.KC2 && ok; ++cc) copy(false);
      tc_commit(&drained[kMmaWarps + c]);
      wait_own(cx, &drained[kMmaWarps + c], 0);
    }
  } else if (warp == kGatherWarp) {
    // ------------------------------- activation gather (FC1), hidden loader (FC2)
    int n = 0, slot = 0, cu = -1;
    uint32_t phase = 0;
    int tok_code = -1, tok_scale = -1;
    bool ok = true;
    for (int hf = 0; hf < 2; ++hf)
    for (Fc1Cursor cur(f0[hf], g); cur.s < f1[hf] && ok; cur.next(g)) {
      if (cur.u != cu) {
        // Lane l gathers row l / (32 / R) of the image and the scales of row l.
        const int pc = unit_row_of<R>(a, xc, cur.u, lane / (32 / R));
        const int ps = unit_row_of<R>(a, xc, cur.u, lane % R);
        tok_code = pc >= 0 ? (pc >> 4) : -1;
        tok_scale = ps >= 0 ? (ps >> 4) : -1;
        cu = cur.u;
      }
      if (n >= S) {
        bool freed = true;
        if (lane == 0) freed = wait_bar(cx, &empty[slot], phase ^ 1);
        if (!(ok = __shfl_sync(0xFFFFFFFFu, freed, 0))) break;
      }
      constexpr int kLanesPerRow = 32 / R, kChunksPerLane = 8 / kLanesPerRow;
      const int r = lane / kLanesPerRow, piece = lane % kLanesPerRow;
      uint8_t* img = ACT + slot * kImage;
      const uint8_t* row = a.plan_codes + static_cast<size_t>(tok_code < 0 ? 0 : tok_code) * g.H +
                           cur.c * kChunkK;
#pragma unroll
      for (int h = 0; h < kChunksPerLane; ++h) {
        const int c16 = piece * kChunksPerLane + h;
        cp_async_16(img + swizzle128(r, c16), row + c16 * 16, tok_code < 0 ? 0u : 16u);
      }
      if (lane < R) {
        const uint8_t* src = a.plan_scales +
                             static_cast<size_t>(tok_scale < 0 ? 0 : tok_scale) * (g.H / kBlock) +
                             cur.c * (kChunkK / kBlock);
        cp_async_4(BSF + slot * L.bsf_stride + lane * 16, src, tok_scale < 0 ? 0u : 4u);
      }
      cp_async_arrive_noinc(&full[slot]);
      ++n;
      if (++slot == S) {
        slot = 0;
        phase ^= 1;
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // Hidden loader: one image per FC2 unit, double-buffered.
    int ordinal = -1;
    cu = -1;
    for (int hf = 0; hf < 2; ++hf)
    for (Fc2Cursor cur(j0[hf], g); cur.j < j1[hf] && ok; cur.next(g)) {
      if (cur.u == cu) continue;
      cu = cur.u;
      ++ordinal;
      const int b = ordinal & 1;
      if (ordinal >= 2) {
        bool freed = true;
        if (lane == 0) freed = wait_bar(cx, &hempty[b], ((ordinal >> 1) - 1) & 1);
        if (!(ok = __shfl_sync(0xFFFFFFFFu, freed, 0))) break;
      }
      // Wait (bounded) for every K chunk of the unit's hidden vector: lane
      // l < KC2 polls chunk l with acquire loads (a short back-off between
      // polls), so all chunks are polled at once; the warp barrier then
      // orders every lane's image loads behind all of the acquires.
      const uint64_t t_start = global_timer_ns();
      const uint32_t* flag = a.hidden_flags + cur.u * g.KC2 + (lane < g.KC2 ? lane : 0);
      for (uint32_t i = 0;; ++i) {
        if (__all_sync(0xFFFFFFFFu, lane >= g.KC2 || load_acquire_gpu(flag) != 0)) break;
        __nanosleep(32);
        if ((i & 7u) == 7u && global_timer_ns() - t_start > a.timeout_ns) {
          if (lane == 0) report(a.status, MOE_ERR_DEVICE_TIMEOUT);
          break;  // proceed with whatever the image holds
        }
      }
      __syncwarp();
      if (lane == 0 && ordinal == 0) MOE_STAMP(9);
      // The image (codes of every K chunk, then their scale atoms) in one
      // batch of independent 16-byte loads per lane: a single L2 round trip.
      if constexpr (R == 8) {
        const uint4* src = reinterpret_cast<const uint4*>(a.hidden + static_cast<size_t>(cur.u) * g.hidden_bytes);
        uint4* codes = reinterpret_cast<uint4*>(HC + b * g.KC2 * kImage);
        uint4* scales = reinterpret_cast<uint4*>(HSF + b * g.KC2 * kScaleAtomBytes);
        const int n_codes = g.KC2 * kActImageBytes / 16, n_all = g.KC2 * kHiddenChunkBytes / 16;
        constexpr int kPerLane = kMaxInterChunks * kHiddenChunkBytes / 16 / 32;
        uint4 v[kPerLane];
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
          const int i = lane + 32 * k;
          if (i < n_all) v[k] = __ldcg(src + i);
        }
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
          const int i = lane + 32 * k;
          if (i < n_codes) codes[i] = v[k];
          else if (i < n_all) scales[i - n_codes] = v[k];
        }
      } else {
        // A pair: rows 0-7 from the first unit's image, rows 8-15 (the
        // second atom of every chunk, bytes 128-255 of every scale atom)
        // from the second's. Per unit: KC2 x 64 code vectors, then the
        // KC2 scale atoms' first 128 bytes (8 vectors each).
        const uint32_t w = xc[cur.u];
        const int first = static_cast<int>(w & kWideFirstMask);
        const int per_unit = g.KC2 * (kActImageBytes / 16 + 8);
        const int n_all = (w >> 31) ? 2 * per_unit : per_unit;
        constexpr int kPerLane = 2 * kMaxInterChunks * (kActImageBytes / 16 + 8) / 32;
        uint4 v[kPerLane];
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
          const int i = lane + 32 * k;
          if (i < n_all) {
            const int half = i >= per_unit, j = i - half * per_unit;
            const uint4* src = reinterpret_cast<const uint4*>(
                a.hidden + static_cast<size_t>(first + half) * g.hidden_bytes);
            const int n_codes = g.KC2 * kActImageBytes / 16;
            v[k] = __ldcg(src + (j < n_codes ? j : n_codes + ((j - n_codes) >> 3) * (kScaleAtomBytes / 16) +
                                                      ((j - n_codes) & 7)));
          }
        }
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
          const int i = lane + 32 * k;
          if (i < n_all) {
            const int half = i >= per_unit, j = i - half * per_unit;
            const int n_codes = g.KC2 * kActImageBytes / 16;
            uint4* dst = j < n_codes
                ? reinterpret_cast<uint4*>(HC + (b * g.KC2 + (j >> 6)) * kImage + half * kActImageBytes) + (j & 63)
                : reinterpret_cast<uint4*>(HSF + (b * g.KC2 + ((j - n_codes) >> 3)) * kScaleAtomBytes + half * 128) +
                      ((j - n_codes) & 7);
            *dst = v[k];
          }
        }
      }
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0 && cur.u != a.withhold_image) mbar_arrive(&hfull[b]);
    }
  } else if (warp >= kEpilogueWarp0 && warp < kEpilogueWarp0 + 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                  // TMEM lane quarter this warp may read
    const int et = tid - kEpilogueWarp0 * 32;
    const int m = q * 32 + lane;             // tile row of this thread
    const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
    const bool fc2_upper_half = g.I > 2 * kBlock;  // issuers 1 and 3 own FC2 K-steps 2-3
    // Unit rows of this CTA's first units, fetched while the first stages stream.
    int* cache_unit = reinterpret_cast<int*>(sm + L.rows);
    int* cache_valid = cache_unit + kRowCache;
    int* cache_first = cache_valid + kRowCache;  // the unit's (first) table unit
    int16_t* cache_rows = reinterpret_cast<int16_t*>(cache_first + kRowCache);
    {
      const int per_unit_fc1 = g.P1 * g.KC1;
      int lo = units, hi = -1;
      for (int h = 0; h < 2; ++h) {
        if (f0[h] < f1[h]) { lo = min(lo, f0[h] / per_unit_fc1); hi = max(hi, (f1[h] - 1) / per_unit_fc1); }
        if (j0[h] < j1[h]) { lo = min(lo, j0[h] / g.NQ); hi = max(hi, (j1[h] - 1) / g.NQ); }
      }
      if (et < kRowCache) {
        const int u = lo + et;
        cache_unit[et] = (u <= hi) ? u : -1;
        cache_first[et] = (u <= hi) ? unit_first_of<R>(xc, u) : -1;
      }
      for (int i = et; i < kRowCache * R; i += 128) {
        const int u = lo + i / R;
        cache_rows[i] = (u <= hi) ? unit_row_of<R>(a, xc, u, i % R) : -1;
      }
      epilogue_sync();
      if (et < kRowCache) {
        int v = 0;
        while (v < R && cache_rows[et * R + v] >= 0) ++v;
        cache_valid[et] = v;
      }
      epilogue_sync();
    }
    auto cached = [&](int u) {
      const int i = u - cache_unit[0];
      return (cache_unit[0] >= 0 && i >= 0 && i < kRowCache && cache_unit[i] == u) ? i : -1;
    };
    auto unit_row = [&](int u, int r) -> int {
      const int i = cached(u);
      return i >= 0 ? cache_rows[i * R + r] : unit_row_of<R>(a, xc, u, r);
    };
    auto unit_first = [&](int u) -> int {
      const int i = cached(u);
      return i >= 0 ? cache_first[i] : unit_first_of<R>(xc, u);
    };
    auto unit_valid = [&](int u) -> int {
      const int i = cached(u);
      if (i >= 0) return cache_valid[i];
      if constexpr (R == 8) {
        return table_unit_valid(a, u);
      } else {
        // A pair's first unit is full: 8 + the second's rows.
        const uint32_t w = xc[u];
        const int first = static_cast<int>(w & kWideFirstMask);
        return table_unit_valid(a, (w >> 31) ? first + 1 : first) + ((w >> 31) ? kUnitRows : 0);
      }
    };
    int k = 0, out_unit = -1, out_pair = -1, out_pair2 = -1, out_valid = 0;
    bool prev_ended = false;
    for (;;) {
      const int set = k % NACC;
      // The metadata and the abort flag are read together, after the wait.
      const bool seen = wait_bar(cx, &accfull[set], (k / NACC) & 1);
      tc_fence_after_sync();
      int4 md = meta[set];
      if (!seen || *cx.abort_flag) {
        if (!epilogue_agree(cx, &accfull[set], (k / NACC) & 1, k, agree)) break;
        tc_fence_after_sync();
        md = meta[set];
      }
      if (md.x == 2) break;
      // The four issuers' accumulators: columns [0, R) tile 0 K-steps 0-1,
      // [R, 2R) tile 0 K-steps 2-3, [2R, 3R) and [3R, 4R) tile 1.
      float v0[R], v1[R], x0[R], x1[R];
      {
        uint32_t rr[R / 2][8];
        const uint32_t base = tmem + lanes + set * RT::kSetColumns;
#pragma unroll
        for (int j = 0; j < R / 2; ++j) tmem_load_8_async(base + 8 * j, rr[j]);
        tmem_wait_loads();
#pragma unroll
        for (int t = 0; t < R; ++t) {
          v0[t] = __uint_as_float(rr[t >> 3][t & 7]);
          x0[t] = __uint_as_float(rr[(R + t) >> 3][t & 7]);
          v1[t] = __uint_as_float(rr[(2 * R + t) >> 3][t & 7]);
          x1[t] = __uint_as_float(rr[(3 * R + t) >> 3][t & 7]);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[set]);
      if (et == 0 && md.x == 0) MOE_STAMP(6);
      ++k;
      if (md.x == 0 || fc2_upper_half) {
#pragma unroll
        for (int t = 0; t < R; ++t) {
          v0[t] += x0[t];
          v1[t] += x1[t];
        }
      }
      if (md.x == 0) {
        // ---- FC1 piece: gate = v0, up = v1 for rows 128p + m.
        const int item = md.y, u = item / g.P1, p = item - u * g.P1;
        const int valid = unit_valid(u);
        if (!(md.z && md.w)) {
          // Split-K: the item's owner is the CTA holding its first stage. Its
          // piece is the last one of its own range, so the other pieces (each
          // the first piece of a later CTA) are usually in L2 by then.
          const int hf = item < items_a ? 0 : 1;
          const int* st = start + hf * (G + 1);
          if (!md.z) {
            // Hand the partial sums to the owner and move on: a CTA owns
            // every item whose first stage it holds, so this is its only
            // hand-off in this half.
            float* dst = a.partials + static_cast<size_t>(cta * 2 + hf) * 2 * R * kTileM;
#pragma unroll
            for (int t = 0; t < R; ++t) {
              if (t >= valid) break;
              dst[t * kTileM + m] = v0[t];
              dst[R * kTileM + t * kTileM + m] = v1[t];
            }
            epilogue_sync();
            if (et == 0) red_release_add_gpu(&a.item_counters[item], 1u);
            continue;
          }
          // The other pieces sit in the CTAs after this one, up to the item's
          // last stage.
          const int item_last = item * g.KC1 + g.KC1 - 1;
          int c_end = cta + 1;
          uint32_t others = 0;
          for (; c_end < G && st[c_end] <= item_last; ++c_end) others += st[c_end] < st[c_end + 1];
          // One thread acquires the count (with a short back-off, so that the
          // polls of many owners do not crowd the counters' L2 lines); the
          // epilogue barrier orders every thread's partial-sum loads after it.
          if (et == 0) {
            const uint64_t t_wait = global_timer_ns();
            for (uint32_t i = 0; load_acquire_gpu(&a.item_counters[item]) < others; ++i) {
              __nanosleep(64);
              if ((i & 15u) == 15u && global_timer_ns() - t_wait > a.timeout_ns) {
                report(a.status, MOE_ERR_DEVICE_TIMEOUT);
                break;
              }
            }
          }
          epilogue_sync();
          if (et == 0) MOE_STAMP(7);
          // Sum the pieces in CTA order, the owner's own piece first; the
          // loads of up to 32 / R pieces are issued together.
          constexpr int kBatch = 32 / R;
          for (int c0 = cta + 1; c0 < c_end; c0 += kBatch) {
            float p0[kBatch][R], p1[kBatch][R];
            bool has[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
              const int c = c0 + j;
              has[j] = c < c_end && st[c] < st[c + 1];
              const float* src = a.partials + static_cast<size_t>(c * 2 + hf) * 2 * R * kTileM;
#pragma unroll
              for (int t = 0; t < R; ++t) {
                const bool ld = has[j] && t < valid;
                p0[j][t] = ld ? __ldcg(src + t * kTileM + m) : 0.f;
                p1[j][t] = ld ? __ldcg(src + R * kTileM + t * kTileM + m) : 0.f;
              }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
              if (!has[j]) continue;
#pragma unroll
              for (int t = 0; t < R; ++t) {
                v0[t] += p0[j][t];
                v1[t] += p1[j][t];
              }
            }
          }
        }
        // SiLU(gate) * up, MXFP8 per 32 hidden values (= this warp's 32 rows).
        if (p * kTileM + q * 32 < g.I) {
          // Row t goes to the hidden image of table unit first + t / 8 (its
          // row t % 8), the layout the read-back decodes.
          const int first = unit_first(u);
          // Rows past `valid` are padding: FC2 reads them but its output
          // columns for them are never stored, so they stay unwritten.
#pragma unroll
          for (int t = 0; t < R; ++t) {
            if (t >= valid) break;
            uint8_t* img = a.hidden + static_cast<size_t>(first + (t >> 3)) * g.hidden_bytes;
            const float h = silu_times(v0[t], v1[t]);
            const float amax = warp_amax(h);
            const int E = mx_exponent(amax, g.floor_rule != 0);
            img[p * kActImageBytes + swizzle128(t & 7, m >> 4) + (m & 15)] = e4m3_code(h * pow2f(-E));
            if (lane == 0)
              img[g.KC2 * kActImageBytes + p * kScaleAtomBytes + scale_atom(t & 7, q)] =
                  static_cast<uint8_t>(E + 127);
          }
        }
        epilogue_sync();
        if (et == 0 && u != a.withhold_unit)
          store_release_gpu(&a.hidden_flags[u * g.KC2 + p], 1u);
        if (et == 0) MOE_STAMP(8);
      } else {
        // ---- FC2 job: rows 256q' + m (v0) and 256q' + 128 + m (v1) -> BF16.
        if (a.early && !prev_ended) {
          // The previous call may write the same output rows: wait for the
          // prep grid's end, which follows the previous experts grid's, and
          // only then let the next call start.
          grid_dependency_wait();
          if (et == 0) grid_launch_dependents();
          prev_ended = true;
        }
        const int j = md.y, u = j / g.NQ, qq = j - u * g.NQ;
        if (u != out_unit) {
          out_pair = unit_row(u, et >> 4);
          if (R == 16) out_pair2 = unit_row(u, 8 + (et >> 4));
          out_valid = unit_valid(u);
          out_unit = u;
        }
        if (out_valid <= 2) {
          // Few rows: no staging; each warp writes its 32 outputs of each row
          // and tile as four 16-byte stores.
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t >= out_valid) break;
            uint16_t* dst = a.out + static_cast<size_t>(unit_row(u, t)) * g.H + qq * 2 * kTileM + q * 32;
            store_row32_bf16(dst, v0[t], lane);
            store_row32_bf16(dst + kTileM, v1[t], lane);
          }
          if (et == 0) MOE_STAMP(12);
          continue;
        }
#pragma unroll
        for (int t = 0; t < R; ++t) {
          OUT[t * 2 * kTileM + m] = __bfloat16_as_ushort(__float2bfloat16_rn(v0[t]));
          OUT[t * 2 * kTileM + kTileM + m] = __bfloat16_as_ushort(__float2bfloat16_rn(v1[t]));
        }
        epilogue_sync();
        // 16 threads per row, two 16-byte stores each; rows 8-15 after 0-7.
#pragma unroll
        for (int half = 0; half < R / 8; ++half) {
          const int pair = half == 0 ? out_pair : out_pair2;
          if (pair < 0) continue;
          const int r = (et >> 4) + 8 * half, ch = et & 15;
          uint16_t* dst = a.out + static_cast<size_t>(pair) * g.H + qq * 2 * kTileM;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int chunk = ch + 16 * h;
            *reinterpret_cast<uint4*>(dst + chunk * 8) =
                *reinterpret_cast<const uint4*>(OUT + r * 2 * kTileM + chunk * 8);
          }
        }
        epilogue_sync();
        if (et == 0) MOE_STAMP(12);
      }
    }
  }

  if (tid == 0) MOE_STAMP(13);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp0) tmem_dealloc(tmem, kTmemColumns);
  if (tid == 0) {
    MOE_STAMP(14);
    span_leave(a.span);
  }
}

// ---------------------------------------------------------------------------
// Cluster variant for calls of one or two tokens, where every unit is one
// expert with at most two rows. One thread-block cluster of C CTAs runs one
// unit: its FC1 stages and FC2 jobs are cut over the cluster's CTAs as the
// kernel above cuts a call's work over the grid (the same Split). Nothing
// goes through global memory between the two GEMMs:
// - a CTA holding a later piece of an FC1 item stores its FP32 partial sums
//   straight into the shared memory of the item's owner (the CTA holding the
//   item's first stage) and arrives on the owner's mbarrier;
// - the owner sums the pieces in CTA order, applies SiLU(gate) * up and the
//   MXFP8 requant into its own hidden-chunk buffer, then sends the chunk to
//   every other CTA of the cluster with shared-to-shared bulk copies counted
//   on their mbarriers. It also writes the chunk to the global hidden image,
//   which moe_copy_hidden reads back.
// The FC2 weights stream into the ring while FC1 is reduced. The host computes
// the per-rank work split (ClusterPlan). Given the routing ids, the producer
// derives its unit from them and starts streaming before the prep grid ends;
// every other warp waits for the prep grid only for what it reads itself.

constexpr int kClusterMaxRows = 2;  // rows of a unit in a call of one or two tokens

// Unit-relative work of CTA `rank` of a C-CTA cluster: FC1 stages [f0, f1)
// (stage s = item * KC1 + chunk) and FC2 jobs [j0, j1).
// FC1 stages and FC2 jobs are each cut evenly over the cluster. FC2 starts
// only once every hidden chunk has landed, so the longest FC1 range sets when
// it starts: balancing FC1 + FC2 stages per CTA instead would lengthen the
// longest FC1 range by the FC2 jobs' unevenness.
struct ClusterRange {
  int f0, f1, j0, j1;
  __host__ __device__ ClusterRange(const Geometry& g, int rank, int C) {
    const int T1 = g.P1 * g.KC1;
    f0 = rank * T1 / C;
    f1 = (rank + 1) * T1 / C;
    j0 = rank * g.NQ / C;
    j1 = (rank + 1) * g.NQ / C;
  }
};

// The owner of FC1 item p (the CTA whose range holds the item's first
// stage), how many later CTAs hold pieces of it, and the piece index of CTA
// `rank` among them (-1 if it holds none).
struct ItemPieces {
  int owner, pieces, slot;
  __host__ __device__ ItemPieces(const Geometry& g, int C, int p, int rank) : owner(-1), pieces(0), slot(-1) {
    const int lo = p * g.KC1, hi = lo + g.KC1;
    for (int r = 0; r < C; ++r) {
      const ClusterRange cr(g, r, C);
      if (cr.f1 <= cr.f0 || cr.f0 >= hi || cr.f1 <= lo) continue;
      if (cr.f0 <= lo) {
        owner = r;
      } else {
        if (r == rank) slot = pieces;
        ++pieces;
      }
    }
  }
};

// Partial sums of one piece in the owner's `out` region: [2 tiles][rows][128].
__host__ __device__ constexpr int cluster_piece_bytes(int rows) { return 2 * rows * kTileM * 4; }

__global__ void __launch_bounds__(kThreads, 1)
    cluster_kernel(const __grid_constant__ ExpertsArgs a, const __grid_constant__ ClusterPlan plan) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const Geometry& g = a.g;
  const Layout L(g.KC2);
  uint8_t* W = sm + L.w;
  uint8_t* ACT = sm + L.act;
  uint8_t* ASF = sm + L.asf;
  uint8_t* HC = sm + L.hcodes;   // the unit's hidden codes, chunk c at c * 1 KB
  uint8_t* HSF = sm + L.hsf;     // their scale atoms, chunk c at c * 512 B
  float* RECV = reinterpret_cast<float*>(sm + L.out);  // partial sums sent to this CTA
  uint8_t* BSF = sm + L.bsf;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + S;
  uint64_t* accfull = empty + S;
  uint64_t* accempty = accfull + NACC;
  uint64_t* recv = accempty + NACC;  // the other pieces of the item this CTA owns
  uint64_t* hidden = recv + 1;       // every chunk of the unit's hidden vector
  uint64_t* drained = hidden + 1;    // [issuer]: its tensor-core work has finished
  int* agree = reinterpret_cast<int*>(sm + L.agree);
  int4* meta = reinterpret_cast<int4*>(sm + L.meta);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + L.misc);  // tmem base, abort

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = static_cast<int>(cluster_ctarank()), u = static_cast<int>(cluster_id_x());
  Ctx cx{&a, reinterpret_cast<volatile uint32_t*>(&misc[1])};
  const int C = plan.C;
  if (tid == 0) {
    span_enter(a.span);
    MOE_STAMP(0);
  }
  struct {
    int f0, f1, j0, j1;
  } cr = {plan.fc1[rank], plan.fc1[rank + 1], plan.fc2[rank], plan.fc2[rank + 1]};
  const int T1 = g.P1 * g.KC1;
  // The item whose first stage this CTA holds (at most one: a range is at
  // most KC1 stages long), and the number of pieces other CTAs send it.
  const int first_item = (cr.f0 + g.KC1 - 1) / g.KC1;
  const bool owns = cr.f1 > cr.f0 && first_item * g.KC1 < cr.f1 && first_item < g.P1;
  const int owned_pieces = owns ? plan.pieces[first_item] : 0;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1 + 32);
      mbar_init(&empty[s], kMmaWarps);
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&accfull[i], kMmaWarps + 1);
      mbar_init(&accempty[i], 4);
    }
    mbar_init(recv, owned_pieces > 0 ? owned_pieces * 128 : 1);  // every epilogue thread of a piece
    mbar_init(hidden, 1 + (owns ? 1 : 0));  // the byte count below + this CTA's own chunk
    misc[1] = 0;
    fence_mbar_init();
    // Chunks from the other owners arrive as bytes.
    mbar_arrive_expect_tx(hidden, (g.P1 - (owns ? 1 : 0)) * kHiddenChunkBytes);
    prefetch_tensormap(&a.wmap);
  } else if (warp == kMmaWarp0 + 1 && lane == 0) {
    for (int i = 0; i < kMmaWarps; ++i) mbar_init(&drained[i], 1);
    for (int i = 0; i < kAgreeSlots; ++i) agree[i] = -1;
    fence_mbar_init();
  }
  for (int i = tid; i < S * kScaleAtomBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(BSF)[i] = make_uint4(0, 0, 0, 0);
  if (warp == kMmaWarp0) {
    tmem_alloc(&misc[0], kTmemColumns);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (tid == 0) MOE_STAMP(16);
  const uint32_t tmem = misc[0];
  // Each warp waits for the prep grid only for what it reads itself: the
  // unit count, and the unit's expert (producer) or rows (gather warp), in
  // one round trip (the table holds min(E, 16B) units, so the reads stay in
  // bounds for every cluster). Given the routing ids, the producer derives
  // the unit count and its expert from them instead (one unit per distinct
  // kept expert, ascending: the canonical table of one or two tokens) and
  // streams weights while the prep grid still runs.
  int units = 0, pre0 = 0, pre1 = 0;
  if (warp == kProducerWarp && a.ids != nullptr) {
    unsigned* bits = reinterpret_cast<unsigned*>(sm + L.table);  // kept experts, E <= 1024 bits
    const int pairs = a.B * kTopK;  // 16 or 32: one pair per lane
    const int e = lane < pairs ? a.ids[lane] : -1;
    bits[lane] = 0;
    const bool valid = lane < pairs && e >= 0 && e < g.E;
    // Kept: the lowest slot of its token with that id (lanes 0-15, 16-31).
    const unsigned in_token = __match_any_sync(0xFFFFFFFFu, valid ? 2 * e + (lane >> 4) : -1 - lane);
    __syncwarp();
    if (valid && __ffs(in_token) - 1 == lane) atomicOr(&bits[e >> 5], 1u << (e & 31));
    __syncwarp();
    // Unit u is the u-th set bit: a prefix count over the words, then the
    // bit inside the word that holds it.
    const unsigned word = bits[lane];
    const int cnt = __popc(word);
    int incl = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int other = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += other;
    }
    units = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const unsigned who = __ballot_sync(0xFFFFFFFFu, u >= incl - cnt && u < incl);
    const int w = who ? __ffs(who) - 1 : 0;
    const int below = __shfl_sync(0xFFFFFFFFu, incl - cnt, w);
    const unsigned ww = __shfl_sync(0xFFFFFFFFu, word, w);
    pre0 = who ? w * 32 + static_cast<int>(__fns(ww, 0, u - below + 1)) : 0;
    if (lane == 0) MOE_STAMP(17);
  } else {
    grid_dependency_wait();
    units = *a.unit_count;
    if (warp == kProducerWarp) {
      pre0 = a.unit_expert[u];
    } else if (warp == kGatherWarp) {
      pre0 = a.unit_rows[u * kUnitRows + (lane >> 2)];
      pre1 = a.unit_rows[u * kUnitRows + (lane & 7)];
      if (lane == 0) MOE_STAMP(3);
    }
  }
  if (u >= units) {  // a cluster without a unit (the same for all its CTAs and warps)
    if (warp == kMmaWarp0) tmem_dealloc(tmem, kTmemColumns);
    if (tid == 0) span_leave(a.span);
    return;
  }
  // Every CTA's barriers are initialised before any CTA of the cluster
  // touches another's shared memory: all threads arrive now, and the
  // epilogue, the only role that reaches into other CTAs, waits before it
  // starts (the other roles wait at the end).
  cluster_arrive();
  if (tid == 0) MOE_STAMP(18);
  const int fc1_stages = T1;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t policy = policy_evict_first();
      const int e = pre0;
      int n = 0, slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      auto issue = [&](int stage, bool stand_in) {
        if (n >= S && !wait_bar(cx, &empty[slot], phase ^ 1)) return false;
        mbar_arrive_expect_tx(&full[slot], kStageWeightBytes + 2 * kScaleAtomBytes);
        if (stand_in) mbar_arrive_count(&full[slot], 32);
        tma_load_3d(W + slot * kStageSmemWeights, &a.wmap, 0, 0, e * g.SPE + stage, &full[slot],
                    policy);
        bulk_load(ASF + slot * 2 * kScaleAtomBytes,
                  a.stages + static_cast<size_t>(e * g.SPE + stage) * kStageBytes + kStageWeightBytes,
                  2 * kScaleAtomBytes, &full[slot], policy);
        if (n == 0) MOE_STAMP(1);
        MOE_STAMP(2);
        ++n;
        if (++slot == S) {
          slot = 0;
          phase ^= 1;
        }
        return true;
      };
      for (int st = cr.f0; st < cr.f1 && ok; ++st) ok = issue(st, false);
      for (int q = cr.j0; q < cr.j1 && ok; ++q)
        for (int c = 0; c < g.KC2 && ok; ++c) ok = issue(fc1_stages + q * g.KC2 + c, true);
      MOE_STAMP_VALUE(15, static_cast<uint64_t>(n));
      if (ok)  // drain, as in the grid kernel
        for (int k = (n > S ? n - S : 0); k < n && ok; ++k) ok = wait_bar(cx, &empty[k % S], (k / S) & 1);
      if (!ok) settle_copies();
    }
  } else if (warp >= kMmaWarp0 && warp < kMmaWarp0 + kMmaWarps) {
    // --------------------------------------------------------- MMA issuers
    if (lane == 0) {
      const int issuer = warp - kMmaWarp0, t = issuer >> 1, k0 = 2 * (issuer & 1);
      const bool lead = issuer == 0;
      const uint32_t hsf_cols = tmem + kTmemHiddenScaleBase + issuer * kHiddenScaleColumns;
      int n = 0, slot = 0, k = 0, first_c = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool fc2_seen = false;
      (void)fc2_seen;
      auto acquire = [&](int set) {
        return k < NACC || wait_bar(cx, &accempty[set], ((k / NACC) - 1) & 1);
      };
      auto advance = [&]() {
        ++n;
        if (++slot == S) {
          slot = 0;
          phase ^= 1;
        }
      };
      for (int st = cr.f0; st < cr.f1 && ok; ++st) {
        const int p = st / g.KC1, c = st - p * g.KC1;
        const bool first = (st == cr.f0) || (c == 0);
        const bool last = (st == cr.f1 - 1) || (c == g.KC1 - 1);
        const int set = k % NACC;
        if (first) {
          if (!(ok = acquire(set))) break;
          first_c = c;
        }
        if (!(ok = wait_bar(cx, &full[slot], phase))) break;
        if (lead && n == 0) MOE_STAMP(4);
        fence_proxy_async_shared();  // the gathered activations were cp.async (generic) writes
        tc_fence_after_sync();
        const uint32_t sf = tmem + kTmemScaleBase + slot * kSlotScaleColumns + issuer * 8;
        tc_copy_scales(sf, desc_scales(ASF + slot * 2 * kScaleAtomBytes + t * kScaleAtomBytes));
        tc_copy_scales(sf + 4, desc_scales(BSF + slot * kScaleAtomBytes));
        const uint64_t dw = desc_sw128(W + slot * kStageSmemWeights + t * (kStageSmemWeights / 2) + k0 * 32);
        const uint64_t dx = desc_sw128(ACT + slot * kActImageBytes + k0 * 32);
        const uint32_t d = tmem + set * kAccSetColumns + issuer * 8;
        tc_mma_mxf8f6f4(d, dw, dx, mma_idesc(k0), sf, sf + 4, first ? 0u : 1u);
        tc_mma_mxf8f6f4(d, dw + 2, dx + 2, mma_idesc(k0 + 1), sf, sf + 4, 1u);
        if (lead) MOE_STAMP(5);
        tc_commit(&empty[slot]);
        advance();
        if (last) {
          if (lead) meta[set] = make_int4(0, u * g.P1 + p, first_c == 0, c == g.KC1 - 1);
          tc_commit(&accfull[set]);
          if (lead) mbar_arrive(&accfull[set]);
          ++k;
        }
      }
      // FC2 reads the whole hidden vector of the unit, sent by the owners.
      if (ok && cr.j0 < cr.j1) {
        ok = wait_bar_cluster(cx, hidden, 0);
        if (lead) MOE_STAMP(9);
        tc_fence_after_sync();
        // The unit's hidden scale atoms, once for all its jobs.
        for (int c = 0; c < g.KC2 && ok; ++c)
          tc_copy_scales(hsf_cols + c * 4, desc_scales(HSF + c * kScaleAtomBytes));
      }
      for (int q = cr.j0; q < cr.j1 && ok; ++q) {
        const int set = k % NACC;
        if (!(ok = acquire(set))) break;
        bool started = false;
        for (int c = 0; c < g.KC2 && ok; ++c) {
          if (!(ok = wait_bar(cx, &full[slot], phase))) break;
          if (lead && !fc2_seen) {
            MOE_STAMP(10);
            fc2_seen = true;
          }
          tc_fence_after_sync();
          const int ksteps = c + 1 < g.KC2 ? 4 : (g.I - c * kChunkK) / kBlock;
          if (k0 < ksteps) {
            const uint32_t sf = tmem + kTmemScaleBase + slot * kSlotScaleColumns + issuer * 8;
            const uint32_t sfh = hsf_cols + c * 4;
            tc_copy_scales(sf, desc_scales(ASF + slot * 2 * kScaleAtomBytes + t * kScaleAtomBytes));
            const uint64_t dw = desc_sw128(W + slot * kStageSmemWeights + t * (kStageSmemWeights / 2) + k0 * 32);
            const uint64_t dh = desc_sw128(HC + c * kActImageBytes + k0 * 32);
            const uint32_t d = tmem + set * kAccSetColumns + issuer * 8;
            tc_mma_mxf8f6f4(d, dw, dh, mma_idesc(k0), sf, sfh, started ? 1u : 0u);
            if (k0 + 1 < ksteps)
              tc_mma_mxf8f6f4(d, dw + 2, dh + 2, mma_idesc(k0 + 1), sf, sfh, 1u);
            started = true;
          }
          if (lead) MOE_STAMP(11);
          tc_commit(&empty[slot]);
          advance();
        }
        if (!ok) break;
        if (lead) meta[set] = make_int4(1, u * g.NQ + q, 0, 0);
        tc_commit(&accfull[set]);
        if (lead) mbar_arrive(&accfull[set]);
        ++k;
      }
      if (lead && ok && !*cx.abort_flag) {  // as in the grid kernel
        const int set = k % NACC;
        if (k < NACC || wait_bar(cx, &accempty[set], ((k / NACC) - 1) & 1)) {
          meta[set] = make_int4(2, 0, 0, 0);
          mbar_arrive_count(&accfull[set], kMmaWarps + 1);
        }
      }
      tc_commit(&drained[issuer]);
      wait_own(cx, &drained[issuer], 0);
    }
  } else if (warp == kGatherWarp) {
    // ------------------------------------------------ activation gather (FC1)
    int n = 0, slot = 0;
    uint32_t phase = 0;
    const int tok_code = pre0 >= 0 ? (pre0 >> 4) : -1;
    const int tok_scale = pre1 >= 0 ? (pre1 >> 4) : -1;
    for (int st = cr.f0; st < cr.f1; ++st) {
      const int c = st % g.KC1;
      if (n >= S) {
        bool freed = true;
        if (lane == 0) freed = wait_bar(cx, &empty[slot], phase ^ 1);
        if (!__shfl_sync(0xFFFFFFFFu, freed, 0)) break;
      }
      const int r = lane >> 2, piece = lane & 3;
      uint8_t* img = ACT + slot * kActImageBytes;
      const uint8_t* row = a.plan_codes + static_cast<size_t>(tok_code < 0 ? 0 : tok_code) * g.H +
                           c * kChunkK;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c16 = piece * 2 + h;
        cp_async_16(img + swizzle128(r, c16), row + c16 * 16, tok_code < 0 ? 0u : 16u);
      }
      if (lane < 8) {
        const uint8_t* src = a.plan_scales +
                             static_cast<size_t>(tok_scale < 0 ? 0 : tok_scale) * (g.H / kBlock) +
                             c * (kChunkK / kBlock);
        cp_async_4(BSF + slot * kScaleAtomBytes + lane * 16, src, tok_scale < 0 ? 0u : 4u);
      }
      cp_async_arrive_noinc(&full[slot]);
      ++n;
      if (++slot == S) {
        slot = 0;
        phase ^= 1;
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp >= kEpilogueWarp0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int et = tid - kEpilogueWarp0 * 32;
    const int m = q * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
    const bool fc2_upper_half = g.I > 2 * kBlock;
    int rows[kClusterMaxRows];  // the unit's pair rows (at most two in these calls)
    int valid = 0;
#pragma unroll
    for (int r = 0; r < kClusterMaxRows; ++r) {
      rows[r] = a.unit_rows[u * kUnitRows + r];
      valid += rows[r] >= 0;
    }
    const int stride = cluster_piece_bytes(a.B) / 4;  // floats per piece slot
    cluster_wait();
    int k = 0;
    for (;;) {
      const int set = k % NACC;
      // The metadata and the abort flag are read together, after the wait.
      const bool seen = wait_bar(cx, &accfull[set], (k / NACC) & 1);
      tc_fence_after_sync();
      int4 md = meta[set];
      if (!seen || *cx.abort_flag) {
        if (!epilogue_agree(cx, &accfull[set], (k / NACC) & 1, k, agree)) break;
        tc_fence_after_sync();
        md = meta[set];
      }
      if (md.x == 2) break;
      float v0[8], v1[8], x0[8], x1[8];
      {
        uint32_t r0[8], r1[8], r2[8], r3[8];
        const uint32_t base = tmem + lanes + set * kAccSetColumns;
        tmem_load_8_async(base + 0, r0);
        tmem_load_8_async(base + 8, r1);
        tmem_load_8_async(base + 16, r2);
        tmem_load_8_async(base + 24, r3);
        tmem_wait_loads();
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          v0[t] = __uint_as_float(r0[t]);
          x0[t] = __uint_as_float(r1[t]);
          v1[t] = __uint_as_float(r2[t]);
          x1[t] = __uint_as_float(r3[t]);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[set]);
      if (et == 0 && md.x == 0) MOE_STAMP(6);
      ++k;
      if (md.x == 0 || fc2_upper_half) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          v0[t] += x0[t];
          v1[t] += x1[t];
        }
      }
      if (md.x == 0) {
        // ---- FC1 piece of item p: gate = v0, up = v1 for rows 128p + m.
        const int p = md.y - u * g.P1;
        if (!md.z) {
          // A later piece: into the owner's shared memory, then its barrier.
          const int owner = plan.owner[p], slot = plan.slot[p][rank];
          if (owner >= 0 && slot >= 0) {
            float* slot_base = RECV + slot * stride;
#pragma unroll
            for (int t = 0; t < kClusterMaxRows; ++t) {
              if (t >= valid) break;
              st_cluster_f32(cluster_map(slot_base + t * kTileM + m, owner), v0[t]);
              st_cluster_f32(cluster_map(slot_base + (a.B + t) * kTileM + m, owner), v1[t]);
            }
            // Each thread's arrival releases its own stores.
            mbar_arrive_remote(cluster_map(recv, owner));
          }
          if (et == 0) MOE_STAMP(7);
          continue;
        }
        if (!md.w && owned_pieces > 0) {
          // Sum the other pieces in CTA order, after the owner's own.
          if (wait_bar_cluster(cx, recv, 0)) {
            if (et == 0) MOE_STAMP(7);
            for (int j = 0; j < owned_pieces; ++j) {
              const float* src = RECV + j * stride;
#pragma unroll
              for (int t = 0; t < kClusterMaxRows; ++t) {
                if (t >= valid) break;
                v0[t] += src[t * kTileM + m];
                v1[t] += src[(a.B + t) * kTileM + m];
              }
            }
          }
        }
        // SiLU(gate) * up, MXFP8 per 32 hidden values, into this CTA's chunk p.
        if (p * kTileM + q * 32 < g.I) {
#pragma unroll
          for (int t = 0; t < kClusterMaxRows; ++t) {
            if (t >= valid) break;
            const float h = silu_times(v0[t], v1[t]);
            const float amax = warp_amax(h);
            const int E = mx_exponent(amax, g.floor_rule != 0);
            HC[p * kActImageBytes + swizzle128(t, m >> 4) + (m & 15)] = e4m3_code(h * pow2f(-E));
            if (lane == 0) HSF[p * kScaleAtomBytes + scale_atom(t, q)] = static_cast<uint8_t>(E + 127);
          }
        }
        fence_proxy_async_shared();  // generic writes, read by tensor-core and bulk copies
        epilogue_sync();
        if (et == 0) MOE_STAMP(8);
        if (et == 0 && u != a.withhold_unit) {
          mbar_arrive(hidden);
          for (int d = 0; d < C; ++d) {
            if (d == rank) continue;
            const uint32_t bar = cluster_map(hidden, d);
            bulk_copy_to_peer(cluster_map(HC + p * kActImageBytes, d), HC + p * kActImageBytes,
                              kActImageBytes, bar);
            bulk_copy_to_peer(cluster_map(HSF + p * kScaleAtomBytes, d), HSF + p * kScaleAtomBytes,
                              kScaleAtomBytes, bar);
          }
        }
        // The global hidden image, for read-back.
        uint8_t* img = a.hidden + static_cast<size_t>(u) * g.hidden_bytes;
        if (et < kActImageBytes / 16)
          reinterpret_cast<uint4*>(img + p * kActImageBytes)[et] =
              reinterpret_cast<const uint4*>(HC + p * kActImageBytes)[et];
        else if (et < kActImageBytes / 16 + kScaleAtomBytes / 16)
          reinterpret_cast<uint4*>(img + g.KC2 * kActImageBytes + p * kScaleAtomBytes)[et - kActImageBytes / 16] =
              reinterpret_cast<const uint4*>(HSF + p * kScaleAtomBytes)[et - kActImageBytes / 16];
      } else {
        // ---- FC2 job: rows 256q' + m (v0) and 256q' + 128 + m (v1) -> BF16.
        const int qq = md.y - u * g.NQ;
#pragma unroll
        for (int t = 0; t < kClusterMaxRows; ++t) {
          if (t >= valid) break;
          // Each warp writes its 32 outputs of each tile as four 16-byte stores.
          uint16_t* dst = a.out + static_cast<size_t>(rows[t]) * g.H + qq * 2 * kTileM + q * 32;
          store_row32_bf16(dst, v0[t], lane);
          store_row32_bf16(dst + kTileM, v1[t], lane);
        }
        if (et == 0) MOE_STAMP(12);
      }
    }
  }

  // No other CTA writes into this one's shared memory after the hidden
  // vector is complete (bounded). A CTA that gave up on it tells the others,
  // after the start-up barrier, so that every CTA of the cluster lets the
  // copies between them land before it exits.
  bool gave_up = false;
  if (tid == 0) gave_up = *cx.abort_flag || !wait_bar_cluster(cx, hidden, 0);
  if (warp < kEpilogueWarp0) cluster_wait();  // the start-up barrier
  if (gave_up)
    for (int d = 0; d < C; ++d) st_cluster_u32(cluster_map(&misc[1], d), 1u);
  if (tid == 0) MOE_STAMP(13);
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  tc_fence_after_sync();
  if (tid == 0 && *cx.abort_flag) settle_copies();
  if (warp == kMmaWarp0) tmem_dealloc(tmem, kTmemColumns);
  if (tid == 0) {
    MOE_STAMP(14);
    span_leave(a.span);
  }
}

}  // namespace

int experts_smem_bytes(const Geometry& g, int unit_rows) { return Layout(g.KC2, unit_rows, true).bytes; }

int experts_max_smem_bytes(const Geometry& g) {
  const int sizes[] = {Layout(g.KC2, 8, true).bytes, Layout(g.KC2, 16, true).bytes, Layout(g.KC2).bytes};
  int m = 0;
  for (int b : sizes) m = b > m ? b : m;
  return m;
}

bool experts_layout_aligned(const Geometry& g) {
  return Layout(g.KC2, 8, true).aligned() && Layout(g.KC2, 16, true).aligned() && Layout(g.KC2).aligned();
}

namespace {
int g_resident_clusters[9] = {};  // clusters of this many CTAs resident at once (0: none)
}

cudaError_t experts_configure(const Geometry& g) {
  // The attribute belongs to the kernel, not to a handle: allow the largest
  // layout any handle can need (I = 512), so every prepared layer launches.
  (void)g;
  const int bytes = Layout(kMaxInterChunks).bytes;  // the cluster variant's
  cudaError_t e = cudaFuncSetAttribute(experts_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Layout(kMaxInterChunks, 8, true).bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(experts_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Layout(kMaxInterChunks, 16, true).bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  e = small_configure();
  if (e != cudaSuccess) return e;
  for (int C = 2; C <= 8; ++C) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int clusters = 0;
    const cudaError_t q = cudaOccupancyMaxActiveClusters(&clusters, cluster_kernel, &cfg);
    g_resident_clusters[C] = q == cudaSuccess ? clusters : 0;
    if (q != cudaSuccess) cudaGetLastError();  // the grid kernel serves these calls then
  }
  return cudaSuccess;
}

// The largest cluster (at most 8 CTAs) of which one per possible unit is
// resident at once, and whose work split the cluster kernel supports: each
// CTA's FC1 range holds at most one item start, and the later pieces of
// every item fit the owner's 4 KB receive region.
int cluster_size_for(const Geometry& g, int batch) {
  if (batch > kClusterMaxRows) return 0;
  const int max_units = g.E < batch * kTopK ? g.E : batch * kTopK;
  for (int C = 8; C >= 2; --C) {
    if (g_resident_clusters[C] < max_units) continue;
    bool ok = true;
    for (int r = 0; r < C && ok; ++r) {
      const ClusterRange cr(g, r, C);
      ok = cr.f1 - cr.f0 <= g.KC1;
    }
    for (int p = 0; p < g.P1 && ok; ++p) {
      const ItemPieces ip(g, C, p, -1);
      ok = ip.owner >= 0 && ip.pieces * cluster_piece_bytes(batch) <= kUnitRows * 2 * kTileM * 2;
    }
    if (ok) return C;
  }
  return 0;
}

cudaError_t experts_occupancy(const Geometry& g, int* blocks_per_sm) {
  int wide = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, experts_kernel<8>, kGridThreads,
                                                                experts_smem_bytes(g, 8));
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&wide, experts_kernel<16>, kGridThreads,
                                                      experts_smem_bytes(g, 16));
  if (e == cudaSuccess && wide < *blocks_per_sm) *blocks_per_sm = wide;
  return e;
}

cudaError_t launch_experts(const ExpertsArgs& a, int grid, cudaStream_t stream, bool pdl,
                           int path, bool small) {
  if (small && a.ids != nullptr && a.B <= kSmallMaxBatch)  // small: the path serves this call
    return launch_small(a, grid, stream, pdl);
  // Calls of more than 8 tokens run 16-row units (pairs of the table's units).
  const int rows = a.B > kUnitRows ? 16 : 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = experts_smem_bytes(a.g, rows);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  const int C = path == kPathCluster ? cluster_size_for(a.g, a.B) : 0;
  if (C > 0) {
    // One cluster per possible unit: at most min(E, 16B) in these calls.
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = C;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
    cfg.numAttrs = n;
    cfg.dynamicSmemBytes = Layout(a.g.KC2).bytes;
    const int max_units = a.g.E < a.B * kTopK ? a.g.E : a.B * kTopK;
    cfg.gridDim = dim3(max_units * C);
    ClusterPlan plan = {};
    plan.C = C;
    for (int r = 0; r <= C; ++r) {
      const ClusterRange cr(a.g, r < C ? r : C - 1, C);
      plan.fc1[r] = r < C ? cr.f0 : cr.f1;
      plan.fc2[r] = r < C ? cr.j0 : cr.j1;
    }
    for (int p = 0; p < a.g.P1; ++p) {
      for (int r = 0; r < 8; ++r) plan.slot[p][r] = -1;
      for (int r = 0; r < C; ++r) {
        const ItemPieces ip(a.g, C, p, r);
        plan.owner[p] = ip.owner;
        plan.pieces[p] = ip.pieces;
        plan.slot[p][r] = static_cast<int8_t>(ip.slot);
      }
    }
    return cudaLaunchKernelEx(&cfg, cluster_kernel, a, plan);
  }
  cfg.numAttrs = n;
  cfg.blockDim = dim3(kGridThreads);
  if (rows == 16) return cudaLaunchKernelEx(&cfg, experts_kernel<16>, a);
  return cudaLaunchKernelEx(&cfg, experts_kernel<8>, a);
}

}  // namespace moe
