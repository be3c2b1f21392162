// Kernel 3 (+4) for calls of one or two tokens: the small-batch experts kernel.
//
// Pages: ...cutedsl.moe.experts (ExpertsKernel: the TMA producer warp, the
// block-scaled FC1/FC2 tcgen05 stages, store_hidden, the hidden exchange
// (ExpertsKernel.partials / load_hidden), fc2 output rows) and
// ...cutedsl.moe.experts_runtime (PersistentExperts: one persistent grid).
//
// The persistent grid kernel's roles, ring, MMAs and work split (FC1 stages
// and FC2 jobs each cut evenly over one CTA per SM), with two changes that
// suit a call of at most 32 (token, slot) pairs:
//   - A call on device buffers is this one launch: no prep grid runs before
//     it (calls on host buffers keep the prep grid, which reads x once, and
//     gather its plan). Every CTA
//     derives the unit table from the routing ids itself (warp 0: one pair
//     per lane; a unit per distinct kept expert, experts ascending, rows in
//     token order: the canonical table), so the producer streams weights
//     from the kernel's first microsecond, and the activation warp quantizes
//     the x chunks it needs to MXFP8 itself. For read-back, CTA 0 writes the
//     unit table and the kept-pair flags and CTA c the plan of K chunk c.
//   - Consecutive launches overlap (programmatic dependent launch): each
//     launch lets the next one start as its CTAs leave, and every role waits
//     for the previous launch to end before it writes global memory that the
//     previous launch reads or writes.
//   - The FC1 -> FC2 hand-off takes one trip through L2 instead of two. Every
//     piece of an FC1 item (a run of its K stages on one CTA) stores its FP32
//     partial sums and release-increments one count per consumer of its
//     unit; there is no owner. Every CTA that runs FC2 jobs of a unit polls
//     its own counts of the unit's items (and sets them back to zero), sums
//     the pieces itself in CTA order (so every consumer gets the same bits),
//     applies SiLU(gate) * up and the MXFP8 requant, and writes the hidden
//     image straight into its own shared memory.
// The warp roles: warp 0 TMA producer, warps 1-4 MMA issuers, warp 5 the
// activations (FC1), warps 6-9 the epilogue (FC1 partial sums; the hidden
// images of this CTA's FC2 units; BF16 output rows).
#include "pipeline.cuh"

namespace moe {
namespace {

constexpr int kSmallMaxUnits = 2 * kTopK;  // distinct experts of two tokens
constexpr int kSmallPieces = 4;            // FC1 pieces one CTA may hold (partials slots)
constexpr int kSmallHidden = 2;            // FC2 units one CTA may serve
constexpr int kSmallUnitPieces = 160;      // FC1 pieces of one unit (<= grid + 4)

// The unit table of the call, in shared memory (after the FC1 range-start
// region of Layout::table, which this kernel does not use).
struct SmallUnits {
  int count;
  int expert[kSmallMaxUnits];
  int row[kSmallMaxUnits][2];   // pair t * 16 + s, -1 padding
  int valid[kSmallMaxUnits];
  unsigned bits[MOE_MAX_EXPERTS / 32];  // kept experts
  unsigned kept;                        // bit p: pair p got a unit row
};

// The FC1 pieces of one FC2 unit of this CTA, in item order and CTA order
// within an item: (item of the unit) << 16 | partial-sum slot. Built at the
// start, off the critical path.
struct SmallPieces {
  int n;
  int entry[kSmallUnitPieces];
};

// Warp 0: the canonical unit table of <= 32 pairs. Pair p = lane; a pair is
// kept when its id is in [0, E) and no lower slot of its token has the same
// id. Unit u is the u-th kept expert in ascending order; its rows are its
// pairs in token order.
__device__ void derive_units(const ExpertsArgs& a, SmallUnits* su, int lane, int e) {
  const int pairs = a.B * kTopK;  // 16 or 32
  su->bits[lane] = 0;
  su->row[lane][0] = -1;
  su->row[lane][1] = -1;
  const bool valid = lane < pairs && e >= 0 && e < a.g.E;
  const unsigned in_token = __match_any_sync(0xFFFFFFFFu, valid ? 2 * e + (lane >> 4) : -1 - lane);
  const bool kept = valid && __ffs(in_token) - 1 == lane;
  const unsigned kept_mask = __ballot_sync(0xFFFFFFFFu, kept);
  __syncwarp();
  if (kept) atomicOr(&su->bits[e >> 5], 1u << (e & 31));
  __syncwarp();
  const unsigned word = su->bits[lane];
  const int cnt = __popc(word);
  int incl = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int other = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += other;
  }
  const int units = __shfl_sync(0xFFFFFFFFu, incl, 31);
  int k = incl - cnt;
  for (unsigned w = word; w != 0; w &= w - 1, ++k) su->expert[k] = lane * 32 + __ffs(w) - 1;
  // Rows: the unit of a kept pair is its expert's rank; the row within the
  // unit is the number of lower lanes (lower tokens) with the same expert.
  const int we = kept ? (e >> 5) : 0;
  const int below = __shfl_sync(0xFFFFFFFFu, incl - cnt, we);
  const unsigned same = __match_any_sync(0xFFFFFFFFu, kept ? e : -1 - lane);
  if (kept) {
    const int u = below + __popc(su->bits[we] & ((1u << (e & 31)) - 1u));
    const int r = __popc(same & ((1u << lane) - 1u));
    su->row[u][r] = lane;
  }
  __syncwarp();
  if (lane < units) su->valid[lane] = (su->row[lane][0] >= 0) + (su->row[lane][1] >= 0);
  if (lane == 0) {
    su->count = units;
    su->kept = kept_mask;
  }
}

// The activation image of one FC1 stage: lane l quantizes values 4l..4l+3 of
// the 128-value K chunk of each valid row (MXFP8: the 8 lanes of a 32-block
// combine their maxima, ceil-rule E8M0 scale, e4m3 codes) and stores them in
// the 128B-swizzled image and the scale atom of the stage's slot.
__device__ __forceinline__ void quantize_rows(const uint2 (&xv)[2], const int (&tok)[2], uint8_t* img,
                                              uint8_t* atom, int lane) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (tok[r] < 0) continue;  // the same for every lane
    const uint32_t w[2] = {xv[r].x, xv[r].y};
    float v[4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
    const int E = mx_exponent(amax, false);
    const float inv = pow2f(-E);
    uint32_t codes = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) codes |= static_cast<uint32_t>(e4m3_code(v[i] * inv)) << (8 * i);
    *reinterpret_cast<uint32_t*>(img + swizzle128(r, lane >> 2) + (lane & 3) * 4) = codes;
    if ((lane & 7) == 0) atom[scale_atom(r, lane >> 3)] = static_cast<uint8_t>(E + 127);
  }
}

// The CTAs that run FC2 jobs of unit u (those holding jobs u * NQ ..
// u * NQ + NQ - 1 with a non-empty range): every one of them reads every
// FC1 piece of the unit.
__device__ __forceinline__ int unit_consumers(const Split& sp, const Geometry& g, int u, int G) {
  const uint32_t J = static_cast<uint32_t>(sp.J), GG = static_cast<uint32_t>(G);
  auto job_owner = [&](int j) {  // the largest c with floor(c * J / G) <= j
    const int c = static_cast<int>((static_cast<uint32_t>(j + 1) * GG - 1u) / J);
    return c < G - 1 ? c : G - 1;
  };
  int n = 0;
  for (int k = job_owner(u * g.NQ); k <= job_owner(u * g.NQ + g.NQ - 1); ++k)
    n += sp.fc2_begin(k + 1) > sp.fc2_begin(k);
  return n;
}

__global__ void __launch_bounds__(kThreads, 1) small_kernel(const __grid_constant__ ExpertsArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const Geometry& g = a.g;
  const Layout L(g.KC2);
  uint8_t* W = sm + L.w;
  uint8_t* ACT = sm + L.act;
  uint8_t* ASF = sm + L.asf;
  uint8_t* HC = sm + L.hcodes;
  uint8_t* BSF = sm + L.bsf;
  uint8_t* HSF = sm + L.hsf;
  SmallUnits* su = reinterpret_cast<SmallUnits*>(sm + L.table);
  SmallPieces* pl = reinterpret_cast<SmallPieces*>(su + 1);  // [kSmallHidden]
  // FC1 range start and first item of CTAs 0..G (the output-staging region,
  // which this kernel does not use).
  uint32_t* span_tbl = reinterpret_cast<uint32_t*>(sm + L.out);  // [kMaxGrid + 1]
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + S;
  uint64_t* accfull = empty + S;
  uint64_t* accempty = accfull + NACC;
  uint64_t* hfull = accempty + NACC;
  uint64_t* drained = hfull + 4;  // [issuer] (hfull + 2 hempty words: Layout's barrier count)
  int* agree = reinterpret_cast<int*>(sm + L.agree);
  int4* meta = reinterpret_cast<int4*>(sm + L.meta);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + L.misc);  // tmem base, abort

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  Ctx cx{&a, reinterpret_cast<volatile uint32_t*>(&misc[1])};

  // The routing ids first: everything the producer streams depends on them.
  int my_id = -1;
  if (warp == kProducerWarp && lane < a.B * kTopK) my_id = a.ids[lane];
  if (tid == 0) {
    span_enter(a.span);
    MOE_STAMP(0);
    // The next launch may start as this one's CTAs leave their SMs.
    grid_launch_dependents();
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1 + 32);       // producer (with bytes) + 32 gather lanes or a stand-in
      mbar_init(&empty[s], kMmaWarps);   // one commit per issuer
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&accfull[i], kMmaWarps + 1);  // issuer commits + the metadata arrival
      mbar_init(&accempty[i], 4);             // one per epilogue warp
    }
    for (int b = 0; b < kSmallHidden; ++b) mbar_init(&hfull[b], 1);
    misc[1] = 0;
    fence_mbar_init();
    prefetch_tensormap(&a.wmap);
  } else if (warp == kMmaWarp0 + 1 && lane == 0) {
    // Bring every cache line of the kernel's parameters in at once.
    asm volatile("" ::"l"(a.stages), "l"(a.hidden), "r"(a.g.SPE), "l"(a.trace), "l"(a.out),
                 "l"(a.timeout_ns));
    for (int i = 0; i < kMmaWarps; ++i) mbar_init(&drained[i], 1);
    for (int i = 0; i < kAgreeSlots; ++i) agree[i] = -1;
    fence_mbar_init();
  }
  if (warp == kProducerWarp) {
    derive_units(a, su, lane, my_id);
    if (lane == 0) MOE_STAMP(17);
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
  const int units = su->count;
  const Split sp(units, g, G);
  const int f0 = sp.fc1_begin(cta), f1 = sp.fc1_begin(cta + 1);
  const int j0 = sp.fc2_begin(cta), j1 = sp.fc2_begin(cta + 1);
  const int fc1_stages = g.P1 * g.KC1;  // FC2 stages follow the FC1 stages of an expert

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      MOE_STAMP(18);
#ifdef MOE_TRACE
      const long long c0 = clock64();
#endif
      const uint64_t policy = policy_evict_first();
#ifdef MOE_TRACE
      MOE_STAMP_VALUE(26, static_cast<uint64_t>(clock64() - c0));
      {
        const long long t0 = clock64();
        const uint64_t gt = global_timer_ns();
        asm volatile("" ::"l"(gt));
        const long long t1 = clock64();
        MOE_STAMP_VALUE(27, static_cast<uint64_t>(t1 - t0));
      }
#endif
      int n = 0, slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      auto issue = [&](int stage, bool stand_in) {
        if (n >= S && !wait_bar(cx, &empty[slot], phase ^ 1)) return false;
        if (n == 0) MOE_STAMP(19);
        mbar_arrive_expect_tx(&full[slot], kStageWeightBytes + 2 * kScaleAtomBytes);
        if (stand_in) mbar_arrive_count(&full[slot], 32);
        tma_load_3d(W + slot * kStageSmemWeights, &a.wmap, 0, 0, stage, &full[slot], policy);
        if (n == 0) MOE_STAMP(20);
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
      for (Fc1Cursor cur(f0, g); cur.s < f1 && ok; cur.next(g))
        ok = issue(su->expert[cur.u] * g.SPE + cur.p * g.KC1 + cur.c, false);
      for (Fc2Cursor cur(j0, g); cur.j < j1 && ok; cur.next(g)) {
        const int base = su->expert[cur.u] * g.SPE + fc1_stages + cur.q * g.KC2;
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
      const uint32_t hsf_cols = tmem + kTmemHiddenScaleBase + issuer * kHiddenScaleColumns;
      int n = 0, slot = 0, k = 0, ordinal = -1, cu = -1, hb = 0, first_c = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool fc2_seen = false;
      (void)fc2_seen;
#ifdef MOE_TRACE
      int fc2_n = 0;
#endif
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
      for (Fc1Cursor cur(f0, g); cur.s < f1 && ok; cur.next(g)) {
        const bool first = (cur.s == f0) || (cur.c == 0);
        const bool last = (cur.s == f1 - 1) || (cur.c == g.KC1 - 1);
        const int set = k % NACC;
        if (first) {
          if (!(ok = acquire(set))) break;
          first_c = cur.c;
        }
        if (!(ok = wait_bar(cx, &full[slot], phase))) break;
        if (lead && n == 0) MOE_STAMP(4);
        fence_proxy_async_shared();  // the activation image was written by generic stores
        tc_fence_after_sync();
        const uint32_t sf = tmem + kTmemScaleBase + slot * kSlotScaleColumns + issuer * 8;
        tc_copy_scales(sf, desc_scales(ASF + slot * 2 * kScaleAtomBytes + t * kScaleAtomBytes));
        tc_copy_scales(sf + 4, desc_scales(BSF + slot * kScaleAtomBytes));
        const uint64_t dw = desc_sw128(W + slot * kStageSmemWeights + t * (kStageSmemWeights / 2) + k0 * 32);
        const uint64_t dx = desc_sw128(ACT + slot * kActImageBytes + k0 * 32);
        const uint32_t d = tmem + set * kAccSetColumns + issuer * 8;
        // Descriptor start addresses count 16-byte units: +2 is the next K-step.
        tc_mma_mxf8f6f4(d, dw, dx, mma_idesc(k0), sf, sf + 4, first ? 0u : 1u);
        tc_mma_mxf8f6f4(d, dw + 2, dx + 2, mma_idesc(k0 + 1), sf, sf + 4, 1u);
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
      for (Fc2Cursor cur(j0, g); cur.j < j1 && ok; cur.next(g)) {
        if (cur.u != cu) {
          ++ordinal;
          hb = ordinal;  // at most kSmallHidden units, one image buffer each
          if (!(ok = wait_bar(cx, &hfull[hb], 0))) break;
          if (lead) MOE_STAMP(9);
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
          if (!(ok = wait_bar(cx, &full[slot], phase))) break;
          if (lead && !fc2_seen) {
            MOE_STAMP(10);
            fc2_seen = true;
          }
          tc_fence_after_sync();
          // K-steps of this chunk: 4, or fewer in the last chunk when I % 128 != 0.
          const int ksteps = c + 1 < g.KC2 ? 4 : (g.I - c * kChunkK) / kBlock;
          if (k0 < ksteps) {
            const uint32_t sf = tmem + kTmemScaleBase + slot * kSlotScaleColumns + issuer * 8;
            const int hc = hb * g.KC2 + c;
            const uint32_t sfh = hsf_cols + hb * 16 + c * 4;
            tc_copy_scales(sf, desc_scales(ASF + slot * 2 * kScaleAtomBytes + t * kScaleAtomBytes));
            const uint64_t dw = desc_sw128(W + slot * kStageSmemWeights + t * (kStageSmemWeights / 2) + k0 * 32);
            const uint64_t dh = desc_sw128(HC + hc * kActImageBytes + k0 * 32);
            const uint32_t d = tmem + set * kAccSetColumns + issuer * 8;
            tc_mma_mxf8f6f4(d, dw, dh, mma_idesc(k0), sf, sfh, started ? 1u : 0u);
            if (k0 + 1 < ksteps)
              tc_mma_mxf8f6f4(d, dw + 2, dh + 2, mma_idesc(k0 + 1), sf, sfh, 1u);
            started = true;
          }
          if (lead) MOE_STAMP(11);
#ifdef MOE_TRACE
          if (lead && fc2_n < 4) MOE_STAMP(28 + fc2_n);
          ++fc2_n;
#endif
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
      // succeeded (as in the grid kernel).
      if (lead && ok && !*cx.abort_flag) {
        const int set = k % NACC;
        if (k < NACC || wait_bar(cx, &accempty[set], ((k / NACC) - 1) & 1)) {
          meta[set] = make_int4(2, 0, 0, 0);
          mbar_arrive_count(&accfull[set], kMmaWarps + 1);
        }
      }
      tc_commit(&drained[issuer]);
      wait_own(cx, &drained[issuer], 0);
    }
  } else if (warp == kGatherWarp && a.x == nullptr) {
    // ------------------------------- activations (FC1), from the prep grid's plan
    // The call's prep grid ran just before (inputs in host memory: it reads
    // x once); each stage's 8 activation rows are gathered from its plan.
    grid_dependency_wait();
    int n = 0, slot = 0, cu = -1;
    uint32_t phase = 0;
    int tok_code = -1, tok_scale = -1;
    for (Fc1Cursor cur(f0, g); cur.s < f1; cur.next(g)) {
      if (cur.u != cu) {
        const int rc = lane >> 2, rs = lane & 7;
        const int pc = rc < 2 ? su->row[cur.u][rc] : -1;
        const int ps = rs < 2 ? su->row[cur.u][rs] : -1;
        tok_code = pc >= 0 ? (pc >> 4) : -1;
        tok_scale = ps >= 0 ? (ps >> 4) : -1;
        cu = cur.u;
      }
      if (n >= S) {
        bool freed = true;
        if (lane == 0) freed = wait_bar(cx, &empty[slot], phase ^ 1);
        if (!__shfl_sync(0xFFFFFFFFu, freed, 0)) break;
      }
      const int r = lane >> 2, piece = lane & 3;
      uint8_t* img = ACT + slot * kActImageBytes;
      const uint8_t* row = a.plan_codes + static_cast<size_t>(tok_code < 0 ? 0 : tok_code) * g.H +
                           cur.c * kChunkK;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c16 = piece * 2 + h;
        cp_async_16(img + swizzle128(r, c16), row + c16 * 16, tok_code < 0 ? 0u : 16u);
      }
      if (lane < 8) {
        const uint8_t* src = a.plan_scales +
                             static_cast<size_t>(tok_scale < 0 ? 0 : tok_scale) * (g.H / kBlock) +
                             cur.c * (kChunkK / kBlock);
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
  } else if (warp == kGatherWarp) {
    // -------------------------------------------- activations (FC1): x -> MXFP8
    // The call is this launch alone: the x chunks of kAhead stages are loaded
    // ahead (one 8-byte load per lane and row), so each stage's image is
    // written as soon as its slot is free. x is an input of the call: no wait
    // for the previous launch.
    constexpr int kAhead = 4;
    const int count = f1 - f0;
    uint2 xv[kAhead][2];
    int tok[kAhead][2];
    auto fetch = [&](int i, int n) {  // ring entry i <- stage f0 + n
      tok[i][0] = tok[i][1] = -1;
      if (n >= count) return;
      const int s = f0 + n, item = s / g.KC1, c = s - item * g.KC1, u = item / g.P1;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int pr = su->row[u][r];
        tok[i][r] = pr >= 0 ? (pr >> 4) : -1;
        if (pr >= 0)
          xv[i][r] = __ldg(reinterpret_cast<const uint2*>(a.x + static_cast<size_t>(pr >> 4) * g.H +
                                                           c * kChunkK) + lane);
      }
    };
#pragma unroll
    for (int i = 0; i < kAhead; ++i) fetch(i, i);
    int slot = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int n0 = 0; n0 < count && ok; n0 += kAhead) {
#pragma unroll
      for (int i = 0; i < kAhead; ++i) {
        const int n = n0 + i;
        if (n >= count) break;
        if (n >= S) {
          bool freed = true;
          if (lane == 0) freed = wait_bar(cx, &empty[slot], phase ^ 1);
          if (!(ok = __shfl_sync(0xFFFFFFFFu, freed, 0))) break;
        }
        quantize_rows(xv[i], tok[i], ACT + slot * kActImageBytes, BSF + slot * kScaleAtomBytes, lane);
        mbar_arrive(&full[slot]);  // each lane's own stores, released to the MMA issuers
        fetch(i, n + kAhead);
        if (++slot == S) {
          slot = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp >= kEpilogueWarp0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                  // TMEM lane quarter this warp may read
    const int et = tid - kEpilogueWarp0 * 32;
    const int m = q * 32 + lane;             // tile row of this thread
    const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
    const bool fc2_upper_half = g.I > 2 * kBlock;  // issuers 1 and 3 own FC2 K-steps 2-3
    const int B = a.B;
    // FC1 pieces this CTA holds: one per item its range touches.
    const int first_item = f0 / g.KC1;
    const int pieces = f1 > f0 ? (f1 - 1) / g.KC1 - first_item + 1 : 0;
    int done = 0;
    // The previous launch may still read or write the buffers below (its
    // partial sums and counts, the plan and unit table, the output): wait for
    // it to end before the first global write.
    grid_dependency_wait();
    // Read-back of the call's inputs as the prep grid would have left them,
    // when no prep grid ran: CTA 0 writes the unit table and the kept-pair
    // flags (and reports dropped pairs), CTA c the MXFP8 plan of K chunk c of
    // every token.
    if (cta == 0 && a.x != nullptr) {
      if (et == 0) *a.unit_count = units;
      for (int i = et; i < units * kUnitRows; i += 128) {
        const int uu = i / kUnitRows, r = i % kUnitRows;
        a.unit_rows[i] = static_cast<int16_t>(r < 2 ? su->row[uu][r] : -1);
      }
      for (int uu = et; uu < units; uu += 128) a.unit_expert[uu] = su->expert[uu];
      const int pairs = B * kTopK;
      if (a.pair_kept != nullptr)
        for (int pp = et; pp < pairs; pp += 128) a.pair_kept[pp] = (su->kept >> pp) & 1u;
      const unsigned all = pairs == 32 ? 0xFFFFFFFFu : (1u << pairs) - 1u;
      if (et == 0 && su->kept != all) report(a.status, MOE_ERR_DEVICE_IDS);
    }
    for (int cc = cta; a.x != nullptr && cc < g.KC1; cc += G) {
      for (int t = 0; t < B; ++t) {
        const float v = __uint_as_float(static_cast<uint32_t>(a.x[static_cast<size_t>(t) * g.H + cc * kChunkK + et]) << 16);
        const int E = mx_exponent(warp_amax(v), false);
        a.plan_codes[static_cast<size_t>(t) * g.H + cc * kChunkK + et] = e4m3_code(v * pow2f(-E));
        if (lane == 0)
          a.plan_scales[static_cast<size_t>(t) * (g.H / kBlock) + cc * (kChunkK / kBlock) + (et >> 5)] =
              static_cast<uint8_t>(E + 127);
      }
    }

    // The FC1 range starts (16 bits) and first items (16 bits) of CTAs 0..G,
    // filled by all epilogue threads at once, so that the piece lists below
    // need no division (a single thread running them with divisions took
    // microseconds).
    for (int c = et; c <= G; c += 128) {
      const int b = sp.fc1_begin(c);
      span_tbl[c] = static_cast<uint32_t>(b) | (static_cast<uint32_t>(b / g.KC1) << 16);
    }
    epilogue_sync();
    // The FC1 pieces behind each FC2 unit of this CTA (at most two units):
    // for every item, the CTAs holding its stages (a binary search over the
    // range starts), in CTA order, skipping CTAs with empty ranges. Epilogue
    // warp w builds the list of unit w.
    if (q == 0 || q == 1) {
      const int ordinal = q, want_unit = j0 / g.NQ + q;
      const bool has = ordinal == 0 ? j1 > j0 : (j1 > j0 && (j1 - 1) / g.NQ >= want_unit);
      if (has && lane == 0) {
        const int u = want_unit;
        auto owner = [&](int st) {  // the largest c with begin(c) <= st
          int lo = 0, hi = G - 1;
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (static_cast<int>(span_tbl[mid] & 0xFFFFu) <= st) lo = mid; else hi = mid - 1;
          }
          return lo;
        };
        SmallPieces& P = pl[ordinal];
        int n = 0;
        for (int p = 0; p < g.P1; ++p) {
          const int item = u * g.P1 + p, s0 = item * g.KC1;
          const int lo = owner(s0), hi = owner(s0 + g.KC1 - 1);
          for (int c = lo; c <= hi; ++c) {
            const uint32_t e0 = span_tbl[c], e1 = span_tbl[c + 1];
            if ((e1 & 0xFFFFu) > (e0 & 0xFFFFu) && n < kSmallUnitPieces)
              P.entry[n++] = (p << 16) | (c * kSmallPieces + (item - static_cast<int>(e0 >> 16)));
          }
        }
        P.n = n;
      }
    }
    if (et == 0) MOE_STAMP(18);
    epilogue_sync();

    // The hidden image of each FC2 unit, built once this CTA's FC1 pieces are
    // out. The partial-sum slots hold a sentinel (a NaN pattern no sum is
    // stored as) until their piece lands, so the sums are their own flags:
    // every piece's loads go out together (16 at a time), and each item's
    // pieces are summed in CTA order: the masked-out terms add -0.0, which
    // leaves every sum (a zero's sign included) unchanged.
    bool built = j1 <= j0;
    int k = 0;
    for (;;) {
      if (!built && done == pieces) {
        built = true;
        int ordinal = 0;
        for (int j = j0; j < j1 && ordinal < kSmallHidden; ++ordinal) {
          const int u = j / g.NQ;
          j = (u + 1) * g.NQ;  // the next unit's first job
          // No abort check here: every epilogue thread must pass the same
          // named barriers, and the build's only waits are bounded polls.
          const SmallPieces& P = pl[ordinal];
          const int valid = su->valid[u];
          uint8_t* hc = HC + ordinal * g.KC2 * kActImageBytes;
          uint8_t* hs = HSF + ordinal * g.KC2 * kScaleAtomBytes;
          if (et == 0) MOE_STAMP(7);
#ifdef MOE_TRACE
          const long long c_start = clock64();
#endif
          // acc[item][gate row 0, gate row 1, up row 0, up row 1]
          float acc[4][4];
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[p][r] = -0.0f;
          // Each thread polls exactly the sums it adds up (rows m of every
          // piece): 16 pieces' loads in flight, then the sentinels among
          // them re-loaded until every sum has landed (bounded).
          const uint64_t t_wait = global_timer_ns();
          for (int e0 = 0; e0 < P.n; e0 += 16) {
            uint32_t v[16][4];
            int pit[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int e = e0 + i;
              const int entry = e < P.n ? P.entry[e] : -1;
              pit[i] = entry >> 16;  // -1 past the end
              const uint32_t* src = a.piece_sums + static_cast<size_t>(entry < 0 ? 0 : (entry & 0xFFFF)) * kSmallPieceWords;
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                const bool ld = entry >= 0 && t < valid;
                v[i][t] = ld ? load_relaxed_gpu(src + t * kTileM + m) : 0x80000000u;
                v[i][2 + t] = ld ? load_relaxed_gpu(src + (B + t) * kTileM + m) : 0x80000000u;
              }
            }
            for (uint32_t poll = 0;; ++poll) {
              bool missing = false;
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int entry = e0 + i < P.n ? P.entry[e0 + i] : -1;
                const uint32_t* src = a.piece_sums + static_cast<size_t>(entry < 0 ? 0 : (entry & 0xFFFF)) * kSmallPieceWords;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                  if (v[i][t] == kPieceSentinel) {
                    missing = true;
                    v[i][t] = load_relaxed_gpu(src + t * kTileM + m);
                  }
                  if (v[i][2 + t] == kPieceSentinel) {
                    missing = true;
                    v[i][2 + t] = load_relaxed_gpu(src + (B + t) * kTileM + m);
                  }
                }
              }
              if (!missing) break;
              if ((poll & 7u) == 7u && global_timer_ns() - t_wait > a.timeout_ns) {
                report(a.status, MOE_ERR_DEVICE_TIMEOUT);
                break;  // go on with whatever landed
              }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
#pragma unroll
              for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[p][r] += pit[i] == p ? __uint_as_float(v[i][r]) : -0.0f;
          }
#ifdef MOE_TRACE
          {
            float sum = 0.f;
#pragma unroll
            for (int p = 0; p < 4; ++p) sum += acc[p][0] + acc[p][2];
            asm volatile("" ::"f"(sum));
            const long long c_loaded = clock64();
            if (et == 0) MOE_STAMP_VALUE(24, static_cast<uint64_t>(c_loaded - c_start));
          }
#endif
          if (et == 0) MOE_STAMP(21);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            if (p >= g.P1 || p * kTileM + q * 32 >= g.I) continue;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (t >= valid) break;
              const float h = silu_times(acc[p][t], acc[p][2 + t]);
              const float amax = warp_amax(h);
              const int E = mx_exponent(amax, g.floor_rule != 0);
              hc[p * kActImageBytes + swizzle128(t, m >> 4) + (m & 15)] = e4m3_code(h * pow2f(-E));
              if (lane == 0) hs[p * kScaleAtomBytes + scale_atom(t, q)] = static_cast<uint8_t>(E + 127);
            }
          }
#ifdef MOE_TRACE
          __syncwarp();
          if (et == 0) MOE_STAMP_VALUE(25, static_cast<uint64_t>(clock64() - c_start));
#endif
          if (et == 0) MOE_STAMP(22);
          fence_proxy_async_shared();  // generic writes, read by the tensor core
          if (et == 0) MOE_STAMP(23);
          epilogue_sync();
          if (et == 0) MOE_STAMP(8);
          if (et == 0 && u != a.withhold_image) mbar_arrive(&hfull[ordinal]);
          // The CTA holding the unit's first FC2 job also writes the image to
          // global memory, for read-back.
          if (j0 <= u * g.NQ) {
            uint8_t* img = a.hidden + static_cast<size_t>(u) * g.hidden_bytes;
            const int n_codes = g.KC2 * kActImageBytes / 16, n_all = g.KC2 * kHiddenChunkBytes / 16;
            for (int i = et; i < n_all; i += 128)
              reinterpret_cast<uint4*>(img)[i] =
                  i < n_codes ? reinterpret_cast<const uint4*>(hc)[i]
                              : reinterpret_cast<const uint4*>(hs)[i - n_codes];
          }
          // This CTA has read every piece of the unit: count it per piece. The
          // unit's last consumer puts the sentinels back and clears the count,
          // so each slot is empty again for the next call (whose pieces are
          // stored only after this launch has ended).
          const int readers = unit_consumers(sp, g, u, G);
          for (int e = et; e < P.n; e += 128) {
            const int slot_index = P.entry[e] & 0xFFFF;
            if (atom_add_acq_rel_gpu(a.piece_readers + slot_index, 1u) + 1u == static_cast<uint32_t>(readers)) {
              uint4* sums = reinterpret_cast<uint4*>(a.piece_sums + static_cast<size_t>(slot_index) * kSmallPieceWords);
              for (int i = 0; i < kSmallPieceWords / 4; ++i)
                sums[i] = make_uint4(kPieceSentinel, kPieceSentinel, kPieceSentinel, kPieceSentinel);
              a.piece_readers[slot_index] = 0u;
            }
          }
        }
      }

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
        // ---- FC1 piece: gate = v0, up = v1 for rows 128p + m -> partial sums.
        const int item = md.y, u = item / g.P1;
        const int valid = su->valid[u];
        // The piece's sums go straight into its slot, which the unit's
        // consumers poll; a sum with the sentinel's bit pattern (a NaN) is
        // stored as the canonical NaN.
        if (u != a.withhold_unit) {
          uint32_t* dst = a.piece_sums + static_cast<size_t>(cta * kSmallPieces + (item - first_item)) * kSmallPieceWords;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t >= valid) break;
            const uint32_t gb = __float_as_uint(v0[t]), ub = __float_as_uint(v1[t]);
            dst[t * kTileM + m] = gb == kPieceSentinel ? 0x7FFFFFFFu : gb;
            dst[(B + t) * kTileM + m] = ub == kPieceSentinel ? 0x7FFFFFFFu : ub;
          }
        }
        ++done;
      } else {
        // ---- FC2 job: rows 256q' + m (v0) and 256q' + 128 + m (v1) -> BF16.
        const int j = md.y, u = j / g.NQ, qq = j - u * g.NQ;
        const int valid = su->valid[u];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (t >= valid) break;
          // Each warp writes its 32 outputs of each tile as four 16-byte stores.
          uint16_t* dst = a.out + static_cast<size_t>(su->row[u][t]) * g.H + qq * 2 * kTileM + q * 32;
          store_row32_bf16(dst, v0[t], lane);
          store_row32_bf16(dst + kTileM, v1[t], lane);
        }
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

}  // namespace

// The small-batch kernel serves a call when it has at most two tokens, the
// layer has at most MOE_MAX_EXPERTS experts (the kept-expert bitmap), and no
// CTA's FC1 range touches more items than it has partial-sum slots for.
bool small_fits(const Geometry& g, int batch, int grid) {
  if (batch > 2 || grid > kMaxGrid || grid + kMaxInterChunks > kSmallUnitPieces) return false;
  static_assert(sizeof(SmallUnits) + kSmallHidden * sizeof(SmallPieces) <= 2 * (kMaxGrid + 1) * 4,
                "the unit table and piece lists fit the table region");
  const int units = g.E < batch * kTopK ? g.E : batch * kTopK;
  for (int n = 1; n <= units; ++n) {
    const Split sp(n, g, grid);
    for (int c = 0; c < grid; ++c) {
      const int a = sp.fc1_begin(c), b = sp.fc1_begin(c + 1);
      if (b > a && (b - 1) / g.KC1 - a / g.KC1 + 1 > kSmallPieces) return false;
      const int j0 = sp.fc2_begin(c), j1 = sp.fc2_begin(c + 1);
      if (j1 > j0 && (j1 - 1) / g.NQ - j0 / g.NQ + 1 > kSmallHidden) return false;
    }
  }
  return true;
}

cudaError_t small_configure() {
  return cudaFuncSetAttribute(small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Layout(kMaxInterChunks).bytes);
}

cudaError_t launch_small(const ExpertsArgs& a, int grid, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Layout(a.g.KC2).bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, small_kernel, a);
}

}  // namespace moe
