// Kernel 3 (+4) for calls of up to eight tokens: the small-batch experts kernel.
//
// Pages: ...cutedsl.moe.experts (ExpertsKernel: the TMA producer warp, the
// block-scaled FC1/FC2 tcgen05 stages, store_hidden, the hidden exchange
// (ExpertsKernel.partials / load_hidden), fc2 output rows) and
// ...cutedsl.moe.experts_runtime (PersistentExperts: one persistent grid;
// `dynamic`: work claimed from a grid-wide counter because the CTAs' stream
// rates differ by microseconds within a call; counters re-armed by call
// parity).
//
// The persistent grid kernel's roles, ring and MMAs, with these changes for a
// call of at most 128 (token, slot) pairs:
//   - A call on device buffers is this one launch: no prep grid runs before
//     it (calls on host buffers keep the prep grid, which reads x once, and
//     copy its plan). Every CTA derives the unit table from the routing ids
//     itself (one pair per thread; a unit per distinct kept expert, experts
//     ascending, rows in token order: the canonical table), and five
//     warps quantize x to MXFP8 once, into a shared-memory image per K chunk
//     that holds every token of the call (the FC1 MMA computes all tokens for
//     each expert; the epilogue keeps the unit's own columns). For
//     read-back, CTA 0 writes the unit table and the kept-pair flags and CTA c
//     the plan of K chunk c.
//   - FC1 is cut into segments (an even share of an item's K chunks, about
//     kSegChunks of them) that the CTAs claim from a counter as their
//     producers get to them, so the CTAs that start first (consecutive
//     launches overlap) take more of the work.
//     FC2 jobs stay split evenly over the CTAs.
//   - The FC1 -> FC2 hand-off takes one trip through L2. Each segment stores
//     its FP32 partial sums into its own slot, whose words hold a sentinel
//     until then; there is no owner and no count to wait for. Every CTA that
//     runs FC2 jobs of a unit polls the sums of all the unit's segments, adds
//     them in segment order (so every consumer gets the same bits), applies
//     SiLU(gate) * up and the MXFP8 requant, and writes the hidden image
//     straight into its own shared memory. The unit's last consumer puts the
//     sentinels back.
//   - Consecutive launches overlap (programmatic dependent launch). The claim
//     counters and segment slots come in two halves that consecutive calls
//     alternate (the host flips the parity per call), so a call's FC1 and
//     hand-off need nothing from the previous call; every write of memory
//     that the previous call reads or writes (the output rows, the read-back
//     copies) waits for the previous call to end, and a CTA lets the next
//     launch start only after that wait, so the call after next finds this
//     call's half at rest.
//   - Two builds (SmallCfg below): calls of one or two tokens take the packed
//     one, whose x and hidden images start 256 bytes apart, which leaves room
//     for a 3-slot weight ring in half an SM; the wide one (2 slots, full
//     8-row images) serves up to eight tokens and the layers too wide for
//     the packed one.
// The warp roles: warp 0 TMA producer, warps 1-4 MMA issuers, warp 5 the
// activations (x quantization; the wait for the previous call; read-back),
// warps 6-9 the epilogue (x quantization first; FC1 segment sums; the hidden
// images of this CTA's FC2 units; BF16 output rows).
#include "pipeline.cuh"

namespace moe {
namespace {

constexpr int kSmallMaxTokens = kSmallMaxBatch;  // tokens of a call (one unit per expert: <= 8 rows)
constexpr int kSmallHidden = 2;            // FC2 units one CTA may serve
constexpr int kXWarps = 5;                 // warps that quantize x: the activation warp + the epilogue
constexpr int kXRaw = 512;                 // wide build: x of chunk c lands at byte 512 of its image (rows 4-7)
// Two CTAs per SM, one of each of two consecutive calls, so that one streams
// while the other hands off and runs its FC2 jobs: each takes at most half of
// the SM's 228 KB of shared memory (less 1 KB reserved per CTA) and half of
// its 512 TMEM columns.
constexpr int kSmemLimit = (233472 - 2 * 1024) / 2;  // dynamic shared memory one CTA may take
constexpr int kSmallTmemColumns = 256;

// The two builds of the kernel:
//   - Wide: a 2-slot weight ring, and for every K chunk a full 8-row image
//     of the call's tokens (an N = 8 MMA reads 8 rows of 128 bytes); up to 8
//     tokens.
//   - Packed: one or two tokens. An MMA still reads 8 rows per K chunk, but
//     only rows 0 and 1 hold tokens, so chunk images start 256 bytes apart
//     and a chunk's rows 2-7 are the next chunks' rows (their output columns
//     are never read). The same for the hidden images and the scale atoms
//     (rows 16 bytes apart: 32 bytes a chunk). That frees the shared memory
//     of a third ring slot. The bytes of a row keep the 128-byte swizzle of
//     their absolute shared-memory address (the pattern a TMA copy writes:
//     16-byte chunk j of the row at address A sits at chunk j ^ (A >> 7) & 7),
//     and the MMA reads them back through a descriptor whose start is the
//     image's (a multiple of 256 bytes) and whose base offset is 0: it
//     swizzles the addresses it forms, as for the K steps inside an atom.
template <int S, bool P>
struct SmallCfg {
  static constexpr int kSlots = S;                                  // weight ring depth
  static constexpr int kMaxUnits = (P ? 2 : kSmallMaxTokens) * kTopK;  // distinct experts of a call
  static constexpr int kImage = P ? 256 : kActImageBytes;          // bytes between chunk images
  static constexpr int kXScale = P ? 32 : kUnitRows * 16;          // bytes between x scale atoms
  static constexpr int kHScale = P ? 32 : kScaleAtomBytes;         // bytes between hidden scale atoms
  static constexpr int kHiddenScaleBase = kTmemScaleBase + S * kSlotScaleColumns;  // 2 units x 16 columns
  static_assert(kHiddenScaleBase + 2 * 16 <= kSmallTmemColumns, "the small kernel's TMEM columns");
  // Byte offset of the 16-byte chunk c16 of row r of image i in a region
  // that starts on a 1024-byte boundary.
  __host__ __device__ static constexpr uint32_t at(int i, int r, int c16) {
    return static_cast<uint32_t>(i * kImage + r * 128) +
           ((static_cast<uint32_t>(c16) ^ (static_cast<uint32_t>(i * kImage / 128 + r) & 7u)) << 4);
  }
};
using WideCfg = SmallCfg<2, false>;
using PackedCfg = SmallCfg<3, true>;

// Stage descriptors, one per ring slot in shared memory: the producer writes
// it before arriving on the slot's full barrier.
constexpr uint32_t kDescSegMask = (1u << 19) - 1u;
constexpr uint32_t kDescFirst = 1u << 27;  // the segment's first chunk: a fresh accumulator
constexpr uint32_t kDescLast = 1u << 28;   // its last chunk: hand the accumulator to the epilogue
constexpr uint32_t kDescEnd = 1u << 29;    // no data: this CTA's FC1 stages are over
__device__ __forceinline__ uint32_t stage_desc(int seg, int c, bool first, bool last) {
  return static_cast<uint32_t>(seg) | (static_cast<uint32_t>(c) << 19) | (first ? kDescFirst : 0u) |
         (last ? kDescLast : 0u);
}

// The unit table of the call, in shared memory: one unit per kept expert
// (at most 8 tokens, so at most 8 rows).
template <int U>
struct SmallUnits {
  int count;
  int expert[U];
  int16_t row[U][kUnitRows];               // pair t * 16 + s of rows 0 .. valid - 1
  uint8_t valid[U];
  uint8_t tokens[U];                       // bit t: token t has a row in the unit
  unsigned bits[MOE_MAX_EXPERTS / 32];     // kept experts
  int below[MOE_MAX_EXPERTS / 32];         // units of the experts in lower words of bits
  unsigned kept[U / 32];                   // bit p % 32 of word p / 32: pair p got a unit row
};

// Shared-memory carve-up of the small kernel (image regions on 1024-byte
// boundaries). An operand read past a region's last image or scale atom
// (the rows and scale rows no token uses) reads the regions after it; the
// end guard keeps every such read inside the allocation. The hand-off lands
// segment sums in the x images and x scales (free once this CTA's FC1 is
// done), plus a pad where half an SM has room for one: enough for all of a
// one-token unit's items at once (kc2 items of small_spi(kc1) segments, a
// gate row and an up row each).
template <class C>
struct SmallLayout {
  int w, asf, hcodes, xc, xs, hsf, table, bars, meta, desc, misc, agree, bytes, land;
  __host__ __device__ static int up(int o, int a) { return (o + a - 1) / a * a; }
  __host__ __device__ SmallLayout(int kc1, int kc2) : SmallLayout(kc1, kc2, 0) {
    const int want = kc2 * small_spi(kc1) * 2 * kTileM * 4 - land;
    if (want > 0) {
      const SmallLayout padded(kc1, kc2, up(want, 16));
      if (padded.bytes <= kSmemLimit) *this = padded;
    }
  }
  __host__ __device__ SmallLayout(int kc1, int kc2, int pad) {
    int o = 0;
    w = o;                    o += C::kSlots * kStageSmemWeights;
    asf = o;                  o += C::kSlots * 2 * kScaleAtomBytes;
    hcodes = o = up(o, 1024); o += kSmallHidden * kc2 * C::kImage;
    xc = o = up(o, 1024);     o += kc1 * C::kImage;
    xs = o = up(o, 16);       o += kc1 * C::kXScale + pad;
    land = o - xc;
    hsf = o = up(o, 16);      o += kSmallHidden * kc2 * C::kHScale;
    table = o = up(o, 16);    o += static_cast<int>(sizeof(SmallUnits<C::kMaxUnits>));
    // full, empty per slot; accfull, accempty per set; hfull per unit;
    // drained per issuer; x ready; previous call done.
    bars = o = up(o, 16);     o += (2 * C::kSlots + 2 * NACC + kSmallHidden + kMmaWarps + 2) * 8;
    meta = o = up(o, 16);     o += NACC * 16;
    desc = o = up(o, 16);     o += C::kSlots * 4;
    misc = o = up(o, 16);     o += 16;
    agree = o = up(o, 16);    o += kAgreeSlots * 4;
    int end = o;
    const int reads[4] = {xc + kc1 * C::kImage + (kActImageBytes - C::kImage),
                          hcodes + kSmallHidden * kc2 * C::kImage + (kActImageBytes - C::kImage),
                          xs + kc1 * C::kXScale + (kScaleAtomBytes - C::kXScale),
                          hsf + kSmallHidden * kc2 * C::kHScale + (kScaleAtomBytes - C::kHScale)};
    for (int r : reads) end = end > r ? end : r;
    bytes = end + 1024;  // slack for aligning the dynamic shared-memory base to 1024
  }
};

// Warps 0 .. nw - 1: the canonical unit table of <= 128 pairs (B <= 8).
// Pair p = 32 * warp + lane; a pair is kept when its id is in [0, E) and no
// lower slot of its token has the same id. Unit u is the u-th kept expert in
// ascending order (at most 8 tokens: one unit per expert); its rows are its
// pairs in token order. `emask` (shared memory, E / 4 words) holds each
// expert's token bits while the table is built.
template <class SU>
__device__ void derive_units(const ExpertsArgs& a, SU* su, uint32_t* emask, int p, int e, int nw) {
  const int pairs = a.B * kTopK, lane = p & 31, warp = p >> 5, E = a.g.E;
  auto sync = [&]() { asm volatile("bar.sync 3, %0;" ::"r"(nw * 32) : "memory"); };
  for (int i = p; i < MOE_MAX_EXPERTS / 32; i += nw * 32) su->bits[i] = 0;
  for (int i = p; i < (E + 3) / 4; i += nw * 32) emask[i] = 0;
  sync();
  const int t = p >> 4;  // the pair's token
  const bool valid = p < pairs && e >= 0 && e < E;
  // A token's 16 pairs share a warp (lanes 0-15 or 16-31).
  const unsigned in_token = __match_any_sync(0xFFFFFFFFu, valid ? 2 * e + (lane >> 4) : -1 - lane);
  const bool kept = valid && __ffs(in_token) - 1 == lane;
  const unsigned kept_mask = __ballot_sync(0xFFFFFFFFu, kept);
  if (lane == 0) su->kept[warp] = kept_mask;
  if (kept) {
    atomicOr(&su->bits[e >> 5], 1u << (e & 31));
    atomicOr(&emask[e >> 2], 1u << ((e & 3) * 8 + t));
  }
  sync();
  if (warp == 0) {
    const unsigned word = su->bits[lane];
    const int cnt = __popc(word);
    int incl = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int other = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += other;
    }
    su->below[lane] = incl - cnt;
    int k = incl - cnt;
    for (unsigned w = word; w != 0; w &= w - 1, ++k) su->expert[k] = lane * 32 + __ffs(w) - 1;
    if (lane == 31) su->count = incl;
  }
  sync();
  if (kept) {
    // The unit of a kept pair is its expert's rank; its row is the number of
    // lower tokens with the same expert.
    const int u = su->below[e >> 5] + __popc(su->bits[e >> 5] & ((1u << (e & 31)) - 1u));
    const unsigned m = (emask[e >> 2] >> ((e & 3) * 8)) & 0xFFu;
    const int r = __popc(m & ((1u << t) - 1u));
    su->row[u][r] = static_cast<int16_t>(p);
    if (r == 0) {
      su->valid[u] = static_cast<uint8_t>(__popc(m));
      su->tokens[u] = static_cast<uint8_t>(m);
    }
  }
}

// MXFP8 of one token row of a 128-value K chunk: lane l quantizes values
// 4l..4l+3 (the 8 lanes of a 32-block combine their maxima, ceil-rule E8M0
// scale, e4m3 codes) into row r of image c of the x images (128B-swizzled)
// and its scale row.
template <class C>
__device__ __forceinline__ void quantize_one(uint2 xv, int r, int c, uint8_t* xc, uint8_t* xs, int lane) {
  const uint32_t w[2] = {xv.x, xv.y};
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
  *reinterpret_cast<uint32_t*>(xc + C::at(c, r, lane >> 2) + (lane & 3) * 4) = codes;
  if ((lane & 7) == 0) xs[c * C::kXScale + scale_atom(r, lane >> 3)] = static_cast<uint8_t>(E + 127);
}

// The CTAs that run FC2 jobs of unit u (those holding jobs u * NQ ..
// u * NQ + NQ - 1 with a non-empty range): every one of them reads every FC1
// segment of the unit.
__device__ __forceinline__ int unit_consumers(const Split& sp, const Geometry& g, int u) {
  int n = 0;
  for (int k = sp.job_owner(u * g.NQ); k <= sp.job_owner(u * g.NQ + g.NQ - 1); ++k)
    n += sp.fc2_begin(k + 1) > sp.fc2_begin(k);
  return n;
}

template <class C>
__global__ void __launch_bounds__(kThreads, 2) small_kernel(const __grid_constant__ ExpertsArgs a) {
  constexpr int S = C::kSlots;
  constexpr bool kPacked = C::kImage < kActImageBytes;
  using Units = SmallUnits<C::kMaxUnits>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const Geometry& g = a.g;
  const SmallLayout<C> L(g.KC1, g.KC2);
  uint8_t* W = sm + L.w;
  uint8_t* XC = sm + L.xc;
  uint8_t* XS = sm + L.xs;
  uint8_t* ASF = sm + L.asf;
  uint8_t* HC = sm + L.hcodes;
  uint8_t* HSF = sm + L.hsf;
  Units* su = reinterpret_cast<Units*>(sm + L.table);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + S;
  uint64_t* accfull = empty + S;
  uint64_t* accempty = accfull + NACC;
  uint64_t* hfull = accempty + NACC;
  uint64_t* drained = hfull + kSmallHidden;  // [issuer]
  uint64_t* xready = drained + kMmaWarps;
  uint64_t* prevdone = xready + 1;
  int* agree = reinterpret_cast<int*>(sm + L.agree);
  int4* meta = reinterpret_cast<int4*>(sm + L.meta);
  volatile uint32_t* sdesc = reinterpret_cast<volatile uint32_t*>(sm + L.desc);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + L.misc);  // tmem base, abort

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  const int B = a.B;
  Ctx cx{&a, reinterpret_cast<volatile uint32_t*>(&misc[1])};
  uint32_t* counters = a.small_counters + 4 * a.parity;  // [0] segments claimed
  const int pw = a.piece_words;  // words per segment slot
  uint32_t* sums = a.piece_sums + static_cast<size_t>(a.parity) * a.seg_cap * pw;
  uint32_t* readers = a.piece_readers + static_cast<size_t>(a.parity) * a.seg_cap;
  const int spi = small_spi(g.KC1);  // segments per item

  // The routing ids and this CTA's first FC1 segment first: everything the
  // producer streams depends on them. The x warps load their chunks of x.
  const int nw = (B * kTopK + 31) / 32;  // warps that derive the unit table (one pair a lane)
  int my_id = -1;
  uint32_t first_claim = 0;
  if (tid < B * kTopK) my_id = a.ids[tid];
  if (tid == 0) first_claim = atomicAdd(counters, 1u);
  const int xw = warp - kGatherWarp;  // x warp 0..4 (warps 5..9)
  // One or two tokens: chunk c's BF16 rows (256 bytes each) go to rows 4-7 of
  // its wide image, which no token uses, or to the packed build's last ring
  // slot, whose first weights the producer loads only once x is quantized.
  auto x_raw = [&](int c) -> uint8_t* {
    return kPacked ? W + (S - 1) * kStageSmemWeights + c * 2 * 2 * kChunkK : XC + c * kActImageBytes + kXRaw;
  };
  if (xw >= 0 && a.x != nullptr && B <= 2 && lane < 16 * B) {
    // Chunk c's BF16 rows, 16 bytes a lane (all in flight).
    const int r = lane >> 4, j = lane & 15;
    for (int c = xw; c < g.KC1; c += kXWarps)
      cp_async_16(x_raw(c) + r * 2 * kChunkK + j * 16, a.x + static_cast<size_t>(r) * g.H + c * kChunkK + j * 8, 16u);
  }
  if (tid == 0) {
    span_enter(a.span);
    MOE_STAMP(0);
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);            // the producer (with the bytes, or a descriptor alone)
      mbar_init(&empty[s], kMmaWarps);   // one commit (or arrival) per issuer
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&accfull[i], kMmaWarps + 1);  // issuer commits + the metadata arrival
      mbar_init(&accempty[i], 4);             // one per epilogue warp
    }
    for (int b = 0; b < kSmallHidden; ++b) mbar_init(&hfull[b], 1);
    mbar_init(xready, kXWarps * 32);
    mbar_init(prevdone, 1);
    misc[1] = 0;
    fence_mbar_init();
    prefetch_tensormap(&a.wmap);
    misc[2] = first_claim;  // every role learns whether this CTA has FC1 work
  } else if (warp == kMmaWarp0 + 1 && lane == 0) {
    // Bring every cache line of the kernel's parameters in at once.
    asm volatile("" ::"l"(a.stages), "l"(a.hidden), "r"(a.g.SPE), "l"(a.trace), "l"(a.out),
                 "l"(a.timeout_ns));
    for (int i = 0; i < kMmaWarps; ++i) mbar_init(&drained[i], 1);
    for (int i = 0; i < kAgreeSlots; ++i) agree[i] = -1;
    fence_mbar_init();
  }
  if (warp < nw) {
    // The experts' token bits (at most 1 KB) go to the hidden images' region
    // and, in the packed build, on into the x images' region: neither is
    // written before the block barrier below.
    derive_units(a, su, reinterpret_cast<uint32_t*>(HC), tid, my_id, nw);
    if (tid == 0) MOE_STAMP(17);
  }
  if (warp == kMmaWarp0) {
    tmem_alloc(&misc[0], kSmallTmemColumns);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (tid == 0) MOE_STAMP(16);
  const uint32_t tmem = misc[0];
  const int units = su->count;
  const int NS = units * g.P1 * spi;  // FC1 segments of the call
  // x images are needed when this CTA runs FC1 segments (its first claim is
  // one) and for the plan read-back of chunk cta.
  const bool need_x = misc[2] < static_cast<uint32_t>(NS) || cta < g.KC1;
  const Split sp(units, g, G);
  const int j0 = sp.fc2_begin(cta), j1 = sp.fc2_begin(cta + 1);
  // This x warp's chunks of x to MXFP8: one or two tokens from the BF16 rows
  // copied at entry; more from registers, the next chunk's rows loading while
  // one is quantized.
  auto quantize_x = [&]() {
    if (B <= 2) {
      for (int c = xw; c < g.KC1; c += kXWarps)
        for (int r = 0; r < B; ++r)
          quantize_one<C>(*reinterpret_cast<const uint2*>(x_raw(c) + r * 2 * kChunkK + lane * 8), r, c, XC, XS, lane);
    } else {
      uint2 cur[kSmallMaxTokens], nxt[kSmallMaxTokens];
      auto load = [&](uint2 (&v)[kSmallMaxTokens], int c) {
#pragma unroll
        for (int r = 0; r < kSmallMaxTokens; ++r)
          if (r < B && c < g.KC1)
            v[r] = __ldg(reinterpret_cast<const uint2*>(a.x + static_cast<size_t>(r) * g.H + c * kChunkK) + lane);
      };
      load(cur, xw);
      for (int c = xw; c < g.KC1; c += kXWarps) {
        load(nxt, c + kXWarps);
#pragma unroll
        for (int r = 0; r < kSmallMaxTokens; ++r)
          if (r < B) quantize_one<C>(cur[r], r, c, XC, XS, lane);
#pragma unroll
        for (int r = 0; r < kSmallMaxTokens; ++r) cur[r] = nxt[r];
      }
    }
    fence_proxy_async_shared();
  };
  const int fc1_stages = g.P1 * g.KC1;  // FC2 stages follow the FC1 stages of an expert

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t policy = policy_evict_first();
      int n = 0, slot = 0, segs = 0;
      uint32_t phase = 0;
      bool ok = true;
      auto issue = [&](int stage, uint32_t desc) {
        if (n >= S && !wait_bar(cx, &empty[slot], phase ^ 1)) return false;
        // The packed build's last slot holds the BF16 rows of x until the
        // x warps have quantized them.
        if (kPacked && n == S - 1 && !wait_bar(cx, xready, 0)) return false;
        sdesc[slot] = desc;
        if (desc == kDescEnd) {
          mbar_arrive(&full[slot]);
        } else {
          if (n == 0) MOE_STAMP(19);
          mbar_arrive_expect_tx(&full[slot], kStageWeightBytes + 2 * kScaleAtomBytes);
          tma_load_3d(W + slot * kStageSmemWeights, &a.wmap, 0, 0, stage, &full[slot], policy);
          bulk_load(ASF + slot * 2 * kScaleAtomBytes,
                    a.stages + static_cast<size_t>(stage) * kStageBytes + kStageWeightBytes,
                    2 * kScaleAtomBytes, &full[slot], policy);
          if (n == 0) MOE_STAMP(1);
          MOE_STAMP(2);
        }
        ++n;
        if (++slot == S) {
          slot = 0;
          phase ^= 1;
        }
        return true;
      };
      // FC1: claimed segments, the next claim in flight while one streams.
      // Claim t is segment NS - 1 - t: the last units' segments go first, so
      // the CTAs that start last (which run the last units' FC2 jobs) find
      // their hidden vectors nearly done, and the CTAs that start first take
      // the first units' segments, which they consume themselves.
      int ticket = static_cast<int>(first_claim);
      while (ok && ticket < NS) {
        const int next = static_cast<int>(atomicAdd(counters, 1u));
        const int seg = NS - 1 - ticket;
        const int item = seg / spi, part = seg - item * spi, u = item / g.P1, pp = item - u * g.P1;
        const int c0 = part * g.KC1 / spi, c1 = (part + 1) * g.KC1 / spi;
        const int base = su->expert[u] * g.SPE + pp * g.KC1;
        for (int c = c0; c < c1 && ok; ++c) ok = issue(base + c, stage_desc(seg, c, c == c0, c == c1 - 1));
        ++segs;
        ticket = next;
      }
      // Each CTA's claims end with one ticket past the segments, so the call
      // takes NS + G tickets; the CTA holding the last one puts the counter
      // back to rest (every other claim of the call is in by then).
      if (ticket == NS + G - 1) *reinterpret_cast<volatile uint32_t*>(counters) = 0u;
      if (ok) ok = issue(0, kDescEnd);
      MOE_STAMP_VALUE(3, static_cast<uint64_t>(segs));
      for (Fc2Cursor cur(j0, g); cur.j < j1 && ok; cur.next(g)) {
        const int base = su->expert[cur.u] * g.SPE + fc1_stages + cur.q * g.KC2;
        for (int c = 0; c < g.KC2 && ok; ++c) ok = issue(base + c, 0u);
      }
      MOE_STAMP_VALUE(15, static_cast<uint64_t>(n));
      // Drain: every issued stage consumed and released before exit.
      if (ok)
        for (int k = (n > S ? n - S : 0); k < n && ok; ++k)
          ok = wait_bar(cx, &empty[k % S], (k / S) & 1);
      if (!ok) settle_copies();
    }
  } else if (warp >= kMmaWarp0 && warp < kMmaWarp0 + kMmaWarps) {
    // --------------------------------------------------------- MMA issuers
    if (lane == 0) {
      const int issuer = warp - kMmaWarp0, t = issuer >> 1, k0 = 2 * (issuer & 1);
      const bool lead = issuer == 0;  // writes the accumulator metadata
      // The hidden scale atoms, copied into TMEM once per unit by the epilogue.
      const uint32_t hsf_cols = tmem + C::kHiddenScaleBase;
      int n = 0, slot = 0, k = 0, ordinal = -1, cu = -1, hb = 0;
      uint32_t phase = 0;
      bool ok = true, have_x = false, fc2_seen = false;
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
      // FC1: the stages of the segments this CTA's producer claimed, in the
      // order of the descriptors, until the end marker.
      for (;;) {
        if (!(ok = wait_bar(cx, &full[slot], phase))) break;
        const uint32_t d = sdesc[slot];
        if (d & kDescEnd) {
          mbar_arrive(&empty[slot]);
          advance();
          break;
        }
        if (!have_x) {
          // The x images are written by generic stores of the x warps.
          if (!(ok = wait_bar(cx, xready, 0))) break;
          fence_proxy_async_shared();
          have_x = true;
        }
        if (lead && n == 0) MOE_STAMP(4);
        const int c = static_cast<int>((d >> 19) & 0xFFu);
        const int set = k % NACC;
        if ((d & kDescFirst) && !(ok = acquire(set))) break;
        tc_fence_after_sync();
        const uint32_t sf = tmem + kTmemScaleBase + slot * kSlotScaleColumns + issuer * 8;
        tc_copy_scales(sf, desc_scales(ASF + slot * 2 * kScaleAtomBytes + t * kScaleAtomBytes));
        tc_copy_scales(sf + 4, desc_scales(XS + c * C::kXScale));
        const uint64_t dw = desc_sw128(W + slot * kStageSmemWeights + t * (kStageSmemWeights / 2) + k0 * 32);
        const uint64_t dx = desc_sw128(XC + c * C::kImage + k0 * 32);
        const uint32_t dt = tmem + set * kAccSetColumns + issuer * 8;
        // Descriptor start addresses count 16-byte units: +2 is the next K-step.
        tc_mma_mxf8f6f4(dt, dw, dx, mma_idesc(k0), sf, sf + 4, (d & kDescFirst) ? 0u : 1u);
        tc_mma_mxf8f6f4(dt, dw + 2, dx + 2, mma_idesc(k0 + 1), sf, sf + 4, 1u);
        if (lead) MOE_STAMP(5);
        tc_commit(&empty[slot]);
        advance();
        if (d & kDescLast) {
          if (lead) meta[set] = make_int4(0, static_cast<int>(d & kDescSegMask), 0, 0);
          tc_commit(&accfull[set]);
          if (lead) mbar_arrive(&accfull[set]);
          ++k;
        }
      }
      // The end of this CTA's FC1 pieces, for the epilogue: an entry with
      // metadata only.
      if (ok) {
        const int set = k % NACC;
        if (lead) {
          if ((ok = acquire(set))) {
            meta[set] = make_int4(3, 0, 0, 0);
            mbar_arrive_count(&accfull[set], kMmaWarps + 1);
          }
        }
        ++k;
      }
      for (Fc2Cursor cur(j0, g); cur.j < j1 && ok; cur.next(g)) {
        if (cur.u != cu) {
          ++ordinal;
          hb = ordinal;  // at most kSmallHidden units, one image buffer each
          if (!(ok = wait_bar(cx, &hfull[hb], 0))) break;
          if (lead) MOE_STAMP(9);
          tc_fence_after_sync();
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
            const uint64_t dh = desc_sw128(HC + hc * C::kImage + k0 * 32);
            const uint32_t dt = tmem + set * kAccSetColumns + issuer * 8;
            tc_mma_mxf8f6f4(dt, dw, dh, mma_idesc(k0), sf, sfh, started ? 1u : 0u);
            if (k0 + 1 < ksteps)
              tc_mma_mxf8f6f4(dt, dw + 2, dh + 2, mma_idesc(k0 + 1), sf, sfh, 1u);
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
  } else if (warp == kGatherWarp) {
    // ------------------------------------------------- activations (FC1)
    uint32_t back_codes[kSmallMaxTokens], back_scales[kSmallMaxTokens];  // plan read-back of chunk cta
    if (a.x != nullptr) {
      // x is an input of the call: quantized without waiting for the
      // previous launch.
      if (B <= 2) {
        cp_async_wait_all();
        __syncwarp();
      }
      if (need_x) quantize_x();
      mbar_arrive(xready);
      if (cta < g.KC1 && wait_bar(cx, xready, 0)) {
        // The plan of chunk cta, read from its image now: the epilogue reuses
        // the images' region once this CTA's FC1 is done.
#pragma unroll
        for (int r = 0; r < kSmallMaxTokens; ++r) {
          if (r >= B) break;
          back_codes[r] = *reinterpret_cast<const uint32_t*>(XC + C::at(cta, r, lane >> 2) + (lane & 3) * 4);
          back_scales[r] = lane < 4 ? XS[cta * C::kXScale + scale_atom(r, lane)] : 0u;
        }
      }
      grid_dependency_wait();
    } else {
      // The call's prep grid ran just before (inputs in host memory: it reads
      // x once): copy its plan of every chunk into the images.
      grid_dependency_wait();
      for (int c = 0; need_x && c < g.KC1; ++c) {
        for (int r0 = 0; r0 < B; r0 += 4) {  // rows r0 .. r0 + 3 of the image, 16 bytes a lane
          const int r = r0 + (lane >> 3), c16 = lane & 7;
          const bool tok = r < B;
          // A packed image's rows past the tokens are the next images' rows.
          if (!kPacked || tok)
            cp_async_16(XC + C::at(c, r, c16),
                        a.plan_codes + static_cast<size_t>(tok ? r : 0) * g.H + c * kChunkK + c16 * 16,
                        tok ? 16u : 0u);
        }
        if (lane < C::kXScale / 16) {
          const bool st = lane < B;
          cp_async_4(XS + c * C::kXScale + lane * 16,
                     a.plan_scales + static_cast<size_t>(st ? lane : 0) * (g.H / kBlock) + c * (kChunkK / kBlock),
                     st ? 4u : 0u);
        }
      }
      cp_async_arrive_noinc(xready);
    }
    // The previous launch has ended: the next one may start as this CTA's
    // work proceeds, and the epilogue may write what the previous launch
    // reads or writes.
    if (lane == 0) {
      MOE_STAMP(18);
      grid_launch_dependents();
      mbar_arrive(prevdone);
    }
    // Read-back of the call's inputs as the prep grid would have left them,
    // when no prep grid ran: CTA 0 writes the unit table and the kept-pair
    // flags (and reports dropped pairs), CTA c the MXFP8 plan of K chunk c of
    // every token (from its image).
    if (a.x != nullptr) {
      if (cta == 0) {
        if (lane == 0) *a.unit_count = units;
        for (int i = lane; i < units * kUnitRows; i += 32) {
          const int uu = i / kUnitRows, r = i % kUnitRows;
          a.unit_rows[i] = static_cast<int16_t>(r < su->valid[uu] ? su->row[uu][r] : -1);
        }
        for (int uu = lane; uu < units; uu += 32) a.unit_expert[uu] = su->expert[uu];
        const int pairs = B * kTopK;
        if (a.pair_kept != nullptr)
          for (int pp = lane; pp < pairs; pp += 32) a.pair_kept[pp] = (su->kept[pp >> 5] >> (pp & 31)) & 1u;
        if (lane < nw) {
          const int left = pairs - 32 * lane;
          const unsigned all = left >= 32 ? 0xFFFFFFFFu : (1u << left) - 1u;
          if (su->kept[lane] != all) report(a.status, MOE_ERR_DEVICE_IDS);
        }
      }
      if (cta < g.KC1) {
#pragma unroll
        for (int r = 0; r < kSmallMaxTokens; ++r) {
          if (r >= B) break;
          *reinterpret_cast<uint32_t*>(a.plan_codes + static_cast<size_t>(r) * g.H + cta * kChunkK + lane * 4) =
              back_codes[r];
          if (lane < 4)
            a.plan_scales[static_cast<size_t>(r) * (g.H / kBlock) + cta * (kChunkK / kBlock) + lane] =
                static_cast<uint8_t>(back_scales[r]);
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
    // Its share of the x chunks first.
    if (a.x != nullptr) {
      if (B <= 2) {
        cp_async_wait_all();
        __syncwarp();
      }
      if (need_x) quantize_x();
    }
    mbar_arrive(xready);
    if (et == 0) MOE_STAMP(28);
    // The previous launch has ended (the activation warp waited for it):
    // false only when this CTA gave up waiting.
    int prev = 0;  // 0: not asked yet, 1: ended, 2: gave up
    auto await_prev = [&]() {
      if (prev == 0) prev = wait_bar(cx, prevdone, 0) ? 1 : 2;
      return prev == 1;
    };

    // The hidden image of each FC2 unit, built once this CTA's FC1 segments
    // are out. The slots hold a sentinel (a NaN pattern no sum is stored as)
    // until their segment lands, so the sums are their own flags: every
    // segment's loads go out together (16 at a time), and each item's
    // segments are summed in order: the masked-out terms add -0.0, which
    // leaves every sum (a zero's sign included) unchanged.
    // A CTA whose first claim found no segment has no FC1 work: its hidden
    // images need only the other CTAs' segments (the end-of-FC1 entry
    // still comes through the accumulator ring, in order).
    bool fc1_over = misc[2] >= static_cast<uint32_t>(NS), built = j1 <= j0;
    int k = 0;
    for (;;) {
      if (!built && fc1_over) {
        built = true;
        wait_bar(cx, xready, 0);  // every x copy has landed before the region is reused
        int ordinal = 0;
        for (int j = j0; j < j1 && ordinal < kSmallHidden; ++ordinal) {
          const int u = j / g.NQ;
          j = (u + 1) * g.NQ;  // the next unit's first job
          // No abort check here: every epilogue thread must pass the same
          // named barriers, and the build's only waits are bounded polls.
          const int valid = su->valid[u];
          const int seg0 = u * g.P1 * spi, nseg = g.P1 * spi;
          const int h0 = ordinal * g.KC2;  // this unit's first hidden image
          if (et == 0) MOE_STAMP(7);
          // The unit's segment sums land in the x images' region (free once
          // this CTA's FC1 MMAs are done and the x copies have landed), a few
          // items at a time: row rr < valid of segment e is the gate of unit
          // row rr, row valid + rr its up. Every 16-byte copy is in flight
          // at once; a copy that brought a sentinel word back is issued again
          // until its segment has landed (bounded).
          float* land = reinterpret_cast<float*>(XC);
          const int rows = 2 * valid;
          const int per_item = spi * rows * kTileM;  // floats of one item's segments
          const int fit = (L.land / 4) / per_item;  // items the region holds (>= 1)
          const int ipb = fit < 4 ? fit : 4;                          // items per landing
          for (int p0 = 0; p0 < g.P1; p0 += ipb) {
            const int p1 = p0 + ipb < g.P1 ? p0 + ipb : g.P1;
            const int copies = (p1 - p0) * spi * rows * (kTileM / 4);
            const uint32_t* from = sums + static_cast<size_t>(seg0 + p0 * spi) * pw;
            auto copy = [&](int i) {  // copy i: segment i / (rows * 32), row (i / 32) % rows, 16 bytes i % 32
              const int e = i / (rows * 32), rr = (i >> 5) - e * rows, c4 = (i & 31) * 4;
              const int row = rr < valid ? rr : B + rr - valid;
              cp_async_16(land + (e * rows + rr) * kTileM + c4,
                          from + static_cast<size_t>(e) * pw + row * kTileM + c4, 16u);
            };
            for (int i = et; i < copies; i += 128) copy(i);
            const uint64_t t_wait = global_timer_ns();
            for (uint32_t poll = 0;; ++poll) {
              cp_async_wait_all();
              bool missing = false;
              for (int i = et; i < copies; i += 128) {
                const uint4 w = *reinterpret_cast<const uint4*>(land + (i >> 5) * kTileM + (i & 31) * 4);
                if (w.x == kPieceSentinel || w.y == kPieceSentinel || w.z == kPieceSentinel || w.w == kPieceSentinel) {
                  missing = true;
                  copy(i);
                }
              }
              if (!missing) {
#ifdef MOE_TRACE
                if (et == 0) MOE_STAMP_VALUE(26, static_cast<uint64_t>(poll));
                if (et == 0) MOE_STAMP(27);
#endif
                break;
              }
              if ((poll & 7u) == 7u && global_timer_ns() - t_wait > a.timeout_ns) {
                report(a.status, MOE_ERR_DEVICE_TIMEOUT);
                cp_async_wait_all();
                break;  // go on with whatever landed
              }
            }
            epilogue_sync();
            if (et == 0) MOE_STAMP(24);
            // Each item's sums in segment order (from -0.0, so a zero's sign
            // is kept), SiLU(gate) * up and the MXFP8 requant of rows m.
            for (int p = p0; p < p1; ++p) {
              if (p * kTileM + q * 32 >= g.I) continue;  // the same for the whole warp
              for (int t = 0; t < valid; ++t) {
                float gate = -0.0f, up = -0.0f;
                const float* src = land + (p - p0) * per_item + m;
#pragma unroll 4
                for (int e = 0; e < spi; ++e) {
                  gate += src[(e * rows + t) * kTileM];
                  up += src[(e * rows + valid + t) * kTileM];
                }
                const float h = silu_times(gate, up);
                const float amax = warp_amax(h);
                const int E = mx_exponent(amax, g.floor_rule != 0);
                HC[C::at(h0 + p, t, m >> 4) + (m & 15)] = e4m3_code(h * pow2f(-E));
                if (lane == 0) HSF[(h0 + p) * C::kHScale + scale_atom(t, q)] = static_cast<uint8_t>(E + 127);
              }
            }
            epilogue_sync();  // the landing is read before the next one overwrites it
          }
          if (et == 0) MOE_STAMP(21);
          fence_proxy_async_shared();  // generic writes, read by the tensor core
          epilogue_sync();
          if (et == 0) MOE_STAMP(8);
          // The unit's hidden scale atoms go into TMEM once, for every issuer;
          // the copies' completion delivers the image.
          if (et == 0 && u != a.withhold_image) {
            tc_fence_after_sync();
            for (int c = 0; c < g.KC2; ++c)
              tc_copy_scales(tmem + C::kHiddenScaleBase + ordinal * 16 + c * 4,
                             desc_scales(HSF + (h0 + c) * C::kHScale));
            tc_commit(&hfull[ordinal]);
          }
          // This CTA has read every segment of the unit: count it per slot.
          // The unit's last consumer puts the sentinels back and clears the
          // count, so the slot is at rest for the call after next.
          const int nreaders = unit_consumers(sp, g, u);
          for (int e = et; e < nseg; e += 128) {
            const int s = seg0 + e;
            if (atom_add_acq_rel_gpu(readers + s, 1u) + 1u == static_cast<uint32_t>(nreaders)) {
              uint4* w = reinterpret_cast<uint4*>(sums + static_cast<size_t>(s) * pw);
              for (int i = 0; i < 2 * B * kTileM / 4; ++i)  // the words this call's tokens use
                w[i] = make_uint4(kPieceSentinel, kPieceSentinel, kPieceSentinel, kPieceSentinel);
              readers[s] = 0u;
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
      if (md.x == 3) {  // this CTA's FC1 segments are all out
        if (et == 0) MOE_STAMP(29);
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty[set]);
        ++k;
        fc1_over = true;
        if (j1 <= j0) break;  // and it has no FC2 job
        continue;
      }
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
        // ---- FC1 segment: gate = v0, up = v1 for rows 128p + m -> its slot.
        // Column j of the accumulator is token j; the slot holds the unit's
        // rows. A sum with the sentinel's bit pattern (a NaN) is stored as
        // the canonical NaN.
        const int seg = md.y, u = seg / (g.P1 * spi);
        if (u != a.withhold_unit) {
          // Token j's column goes to the unit row of token j, if it has one.
          uint32_t* dst = sums + static_cast<size_t>(seg) * pw;
          const unsigned tokens = su->tokens[u];
#pragma unroll
          for (int j = 0; j < kSmallMaxTokens; ++j) {
            if (j >= B) break;
            if (!((tokens >> j) & 1u)) continue;
            const int t = __popc(tokens & ((1u << j) - 1u));
            const uint32_t gb = __float_as_uint(v0[j]), ub = __float_as_uint(v1[j]);
            dst[t * kTileM + m] = gb == kPieceSentinel ? 0x7FFFFFFFu : gb;
            dst[(B + t) * kTileM + m] = ub == kPieceSentinel ? 0x7FFFFFFFu : ub;
          }
        }
      } else {
        // ---- FC2 job: rows 256q' + m (v0) and 256q' + 128 + m (v1) -> BF16,
        // once the previous launch (which may read or write the output) has ended.
        const int j = md.y, u = j / g.NQ, qq = j - u * g.NQ;
        const int valid = await_prev() ? su->valid[u] : 0;
#pragma unroll
        for (int t = 0; t < kUnitRows; ++t) {
          if (t >= valid) break;
          // Each warp writes its 32 outputs of each tile as four 16-byte stores.
          uint16_t* dst = a.out + static_cast<size_t>(su->row[u][t]) * g.H + qq * 2 * kTileM + q * 32;
          store_row32_bf16(dst, v0[t], lane);
          store_row32_bf16(dst + kTileM, v1[t], lane);
        }
        if (et == 0) MOE_STAMP(12);
        if (j == j1 - 1) break;  // this CTA's last FC2 job (the end entry need not be waited for)
      }
    }
    // Read-back of the hidden images: the CTA holding a unit's first FC2 job
    // copies it to global memory.
    if (built && j1 > j0 && await_prev()) {
      int ordinal = 0;
      for (int j = j0; j < j1 && ordinal < kSmallHidden; ++ordinal) {
        const int u = j / g.NQ;
        j = (u + 1) * g.NQ;
        if (j0 > u * g.NQ) continue;
        // In the read-back layout: a full 8-row image per K chunk, then a
        // 512-byte scale atom per chunk (the packed build stores rows 0-1).
        const int h0 = ordinal * g.KC2, rows = kPacked ? 2 : kUnitRows;
        const int per_atom = kPacked ? rows : kScaleAtomBytes / 16;
        uint8_t* img = a.hidden + static_cast<size_t>(u) * g.hidden_bytes;
        const int n_codes = g.KC2 * rows * 8, n_all = n_codes + g.KC2 * per_atom;
        for (int i = et; i < n_all; i += 128) {
          if (i < n_codes) {
            const int p = i / (rows * 8), r = (i >> 3) % rows, c16 = i & 7;
            *reinterpret_cast<uint4*>(img + p * kActImageBytes + swizzle128(r, c16)) =
                *reinterpret_cast<const uint4*>(HC + C::at(h0 + p, r, c16));
          } else {
            const int p = (i - n_codes) / per_atom, v = (i - n_codes) % per_atom;
            *reinterpret_cast<uint4*>(img + g.KC2 * kActImageBytes + p * kScaleAtomBytes + v * 16) =
                *reinterpret_cast<const uint4*>(HSF + (h0 + p) * C::kHScale + v * 16);
          }
        }
      }
    }
  }

  if (tid == 0) MOE_STAMP(13);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp0) tmem_dealloc(tmem, kSmallTmemColumns);
  if (tid == 0) {
    MOE_STAMP(14);
    span_leave(a.span);
  }
}

}  // namespace

namespace {

// Whether build C of the kernel serves calls of `batch` tokens on this layer:
// its shared-memory layout fits half an SM, the hidden build can land one
// item's segments (two rows per token) in the x images' region, the segment
// slots fit the descriptors' field, and no CTA's FC2 jobs span more units
// than it has hidden images for.
template <class C>
bool fits(const Geometry& g, int batch, int grid) {
  if (batch > C::kMaxUnits / kTopK || grid > kMaxGrid || SmallLayout<C>(g.KC1, g.KC2).bytes > kSmemLimit)
    return false;
  const int spi = small_spi(g.KC1);
  if (spi * 2 * batch * kTileM * 4 > SmallLayout<C>(g.KC1, g.KC2).land) return false;
  if (small_seg_cap(g) > static_cast<int>(kDescSegMask)) return false;
  const int units = g.E < batch * kTopK ? g.E : batch * kTopK;
  for (int n = 1; n <= units; ++n) {
    const Split sp(n, g, grid);
    for (int c = 0; c < grid; ++c) {
      const int j0 = sp.fc2_begin(c), j1 = sp.fc2_begin(c + 1);
      if (j1 > j0 && (j1 - 1) / g.NQ - j0 / g.NQ + 1 > kSmallHidden) return false;
    }
  }
  return true;
}

template <class C>
cudaError_t launch(const ExpertsArgs& a, int grid, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SmallLayout<C>(a.g.KC1, a.g.KC2).bytes;
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
  return cudaLaunchKernelEx(&cfg, small_kernel<C>, a);
}

}  // namespace

// The small-batch kernel serves a call of at most eight tokens on a layer of
// at most MOE_MAX_EXPERTS experts (the kept-expert bitmap) when one of its
// builds fits; calls of one or two tokens take the packed build (a 3-slot
// ring) where it fits.
int small_build(const Geometry& g, int batch, int grid) {
  if (fits<PackedCfg>(g, batch, grid)) return kSmallPacked;
  if (fits<WideCfg>(g, batch, grid)) return kSmallWide;
  return 0;
}

bool small_fits(const Geometry& g, int batch, int grid) { return small_build(g, batch, grid) != 0; }

cudaError_t small_configure() {
  cudaError_t e = cudaFuncSetAttribute(small_kernel<WideCfg>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(small_kernel<PackedCfg>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  return e;
}

cudaError_t launch_small(const ExpertsArgs& a, int grid, cudaStream_t stream, bool pdl) {
  if (small_build(a.g, a.B, grid) == kSmallPacked) return launch<PackedCfg>(a, grid, stream, pdl);
  return launch<WideCfg>(a, grid, stream, pdl);
}

}  // namespace moe
