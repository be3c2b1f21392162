// Kernel 3 (+4): the persistent experts kernel with its BF16 output epilogue.
//
// Pages: ...cutedsl.moe.experts (ExpertsKernel: the TMA producer warp, the
// block-scaled FC1/FC2 tcgen05 stages, store_hidden, the hidden exchange,
// fc2 output rows) and ...cutedsl.moe.experts_runtime (PersistentExperts:
// one co-resident persistent grid, per-call workspace).
//
// One CTA per SM, 8 warps:
//   warp 0  TMA producer: one 17 KB stage per ring slot (two 128-row e2m1
//           tiles x 128 K, expanded to 32 KB of 8-bit slots in shared
//           memory with the 128-byte swizzle, plus 1 KB of pre-tiled scales)
//   warp 1  MMA issuer: per stage, copies the scale atoms into TMEM and
//           issues 2 x 4 tcgen05.mma kind::mxf8f6f4.block_scale (M = 128
//           weight rows, N = 8 unit rows, K = 32) into a TMEM accumulator set
//   warp 2  FC1: cp.async gather of each stage's 8 MXFP8 activation rows
//           from the plan; FC2: waits for each unit's hidden vector (bounded)
//           and loads it into shared memory
//   warp 3  TMEM allocation
//   warps 4-7 epilogue: FC1 -> split-K reduction, SiLU(gate) * up, MXFP8
//           hidden requant, publish; FC2 -> BF16 rows with 16-byte stores
//
// Work split: FC1 stages (unit, tile pair, K chunk) and FC2 jobs (unit, 256
// output rows) are cut into contiguous per-CTA ranges of near-equal bytes.
// An FC1 item split across CTAs is reduced by the last CTA to finish its
// piece (an atomic counter; a fixed CTA order keeps the sum deterministic).
// Every wait is bounded by a time limit and reports MOE_ERR_DEVICE_TIMEOUT.
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int S = kRingStages;
constexpr int NACC = kAccSets;

struct Layout {
  int w, act, asf, hcodes, out, bsf, hsf, bars, meta, misc, bytes;
  __host__ __device__ explicit Layout(int kc2) {
    int o = 0;
    w = o;      o += S * kStageSmemWeights;
    act = o;    o += S * kActImageBytes;
    asf = o;    o += S * 2 * kScaleAtomBytes;
    hcodes = o; o += 2 * kc2 * kActImageBytes;
    out = o;    o += kUnitRows * 2 * kTileM * 2;
    bsf = o;    o += S * kScaleAtomBytes;
    hsf = o;    o += 2 * kc2 * kScaleAtomBytes;
    bars = o;   o += (2 * S + 2 * NACC + 4) * 8;
    meta = o;   o += NACC * 16;
    misc = o;   o += 16;
    bytes = o + 1024;  // alignment slack
  }
};

// Per-call split of the work over the grid; every CTA and role computes the
// same function. FC2 jobs are cut evenly; FC1 stages fill each CTA up to an
// equal share of all stages (both kinds stream 17 KB per stage). When the
// shares are too small for that to stay monotone, both are cut evenly.
struct Split {
  int T1, J, KC2, G;
  long long T;
  bool balanced;
  __device__ Split(int units, const Geometry& g, int grid) {
    T1 = units * g.P1 * g.KC1;
    J = units * g.NQ;
    KC2 = g.KC2;
    G = grid;
    T = static_cast<long long>(T1) + static_cast<long long>(J) * KC2;
    balanced = T / G >= static_cast<long long>(KC2) * ((J + G - 1) / G);
  }
  __device__ int fc2_begin(int c) const {
    return static_cast<int>(static_cast<long long>(c) * J / G);
  }
  __device__ int fc1_begin(int c) const {
    if (c >= G) return T1;
    if (!balanced) return static_cast<int>(static_cast<long long>(c) * T1 / G);
    long long v = static_cast<long long>(c) * T / G - static_cast<long long>(KC2) * fc2_begin(c);
    return static_cast<int>(v < 0 ? 0 : (v > T1 ? T1 : v));
  }
  // The CTA whose FC1 range holds stage s (largest c with fc1_begin(c) <= s).
  __device__ int cta_of(int s) const {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (fc1_begin(mid) <= s) lo = mid; else hi = mid - 1;
    }
    return lo;
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
    if (mbar_test(bar, parity)) return true;
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

__device__ __forceinline__ float silu_times(float gate, float up) {
  return gate / (1.0f + expf(-gate)) * up;
}

__device__ __forceinline__ uint64_t desc_sw128(const void* p) {
  return smem_desc(smem_addr(p), 16, 1024, 2);
}
__device__ __forceinline__ uint64_t desc_scales(const void* p) {
  return smem_desc(smem_addr(p), 128, 128, 0);
}

__global__ void __launch_bounds__(kThreads, 1) experts_kernel(const __grid_constant__ ExpertsArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const Geometry& g = a.g;
  const Layout L(g.KC2);
  uint8_t* W = sm + L.w;
  uint8_t* ACT = sm + L.act;
  uint8_t* ASF = sm + L.asf;
  uint8_t* HC = sm + L.hcodes;
  uint16_t* OUT = reinterpret_cast<uint16_t*>(sm + L.out);
  uint8_t* BSF = sm + L.bsf;
  uint8_t* HSF = sm + L.hsf;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + S;
  uint64_t* accfull = empty + S;
  uint64_t* accempty = accfull + NACC;
  uint64_t* hfull = accempty + NACC;
  uint64_t* hempty = hfull + 2;
  int4* meta = reinterpret_cast<int4*>(sm + L.meta);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + L.misc);  // tmem base, abort, last flag

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  Ctx cx{&a, reinterpret_cast<volatile uint32_t*>(&misc[1])};

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1 + 32);  // producer (with bytes) + 32 gather lanes or a stand-in
      mbar_init(&empty[s], 1);      // MMA commit
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&accfull[i], 2);    // MMA commit + metadata arrival
      mbar_init(&accempty[i], 4);   // one per epilogue warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&hfull[b], 1);
      mbar_init(&hempty[b], 1);
    }
    misc[1] = 0;
    misc[2] = 0;
    fence_mbar_init();
    prefetch_tensormap(&a.wmap);
  }
  for (int i = tid; i < S * kScaleAtomBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(BSF)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 3) {
    tmem_alloc(&misc[0], kTmemColumns);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = misc[0];

  // The plan, unit table and cleared counters of the preceding prep grid.
  grid_dependency_wait();
  const int units = *a.unit_count;
  const Split sp(units, g, G);
  const int f0 = sp.fc1_begin(cta), f1 = sp.fc1_begin(cta + 1);
  const int j0 = sp.fc2_begin(cta), j1 = sp.fc2_begin(cta + 1);
  const int fc1_base = g.P1 * g.KC1;  // FC2 stages follow the FC1 stages of an expert

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t policy = policy_evict_first();
      int n = 0;
      bool ok = true;
      auto issue = [&](int stage, bool stand_in) {
        const int slot = n % S;
        const uint32_t phase = (n / S) & 1;
        if (n >= S && !wait_bar(cx, &empty[slot], phase ^ 1)) return false;
        mbar_arrive_expect_tx(&full[slot], kStageWeightBytes + 2 * kScaleAtomBytes);
        if (stand_in) mbar_arrive_count(&full[slot], 32);
        tma_load_3d(W + slot * kStageSmemWeights, &a.wmap, 0, 0, stage, &full[slot], policy);
        bulk_load(ASF + slot * 2 * kScaleAtomBytes,
                  a.stages + static_cast<size_t>(stage) * kStageBytes + kStageWeightBytes,
                  2 * kScaleAtomBytes, &full[slot], policy);
        ++n;
        return true;
      };
      int cu = -1, e = 0;
      for (int s = f0; s < f1 && ok; ++s) {
        const int item = s / g.KC1, c = s % g.KC1, u = item / g.P1, p = item % g.P1;
        if (u != cu) { e = a.unit_expert[u]; cu = u; }
        ok = issue(e * g.SPE + p * g.KC1 + c, false);
      }
      cu = -1;
      for (int j = j0; j < j1 && ok; ++j) {
        const int u = j / g.NQ, q = j % g.NQ;
        if (u != cu) { e = a.unit_expert[u]; cu = u; }
        for (int c = 0; c < g.KC2 && ok; ++c) ok = issue(e * g.SPE + fc1_base + q * g.KC2 + c, true);
      }
      if (ok) {
        // Drain: every issued stage consumed and released before exit.
        for (int k = (n > S ? n - S : 0); k < n; ++k)
          if (!wait_bar(cx, &empty[k % S], (k / S) & 1)) break;
      } else {
        __nanosleep(50000);  // in-flight copies land before the CTA exits
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int n = 0, k = 0, ordinal = -1, cu = -1, hb = 0, first_stage = 0;
      bool ok = true;
      auto acquire = [&](int set) {
        return k < NACC || wait_bar(cx, &accempty[set], ((k / NACC) - 1) & 1);
      };
      for (int s = f0; s < f1 && ok; ++s) {
        const int item = s / g.KC1, c = s % g.KC1;
        const bool first = (s == f0) || (c == 0), last = (s == f1 - 1) || (c == g.KC1 - 1);
        const int set = k % NACC;
        if (first) {
          if (!(ok = acquire(set))) break;
          first_stage = s;
        }
        const int slot = n % S;
        if (!(ok = wait_bar(cx, &full[slot], (n / S) & 1))) break;
        fence_proxy_async_shared();  // the gathered activations were cp.async (generic) writes
        tc_fence_after_sync();
        const uint32_t sf = tmem + kTmemScaleBase + slot * 16;
        const uint8_t* asf = ASF + slot * 2 * kScaleAtomBytes;
        tc_copy_scales(sf + 0, desc_scales(asf));
        tc_copy_scales(sf + 4, desc_scales(asf + kScaleAtomBytes));
        tc_copy_scales(sf + 8, desc_scales(BSF + slot * kScaleAtomBytes));
        const uint8_t* w = W + slot * kStageSmemWeights;
        const uint8_t* x = ACT + slot * kActImageBytes;
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_mxf8f6f4(tmem + set * 16 + t * 8, desc_sw128(w + t * (kStageSmemWeights / 2) + kk * 32),
                            desc_sw128(x + kk * 32), mma_idesc(kk), sf + 4 * t, sf + 8,
                            (first && kk == 0) ? 0u : 1u);
        tc_commit(&empty[slot]);
        ++n;
        if (last) {
          meta[set] = make_int4(0, item, first_stage, s);
          tc_commit(&accfull[set]);
          mbar_arrive(&accfull[set]);
          ++k;
        }
      }
      for (int j = j0; j < j1 && ok; ++j) {
        const int u = j / g.NQ;
        if (u != cu) {
          if (cu >= 0) tc_commit(&hempty[hb]);
          ++ordinal;
          hb = ordinal & 1;
          if (!(ok = wait_bar(cx, &hfull[hb], (ordinal >> 1) & 1))) break;
          tc_fence_after_sync();
          cu = u;
        }
        const int set = k % NACC;
        if (!(ok = acquire(set))) break;
        for (int c = 0; c < g.KC2 && ok; ++c) {
          const int slot = n % S;
          if (!(ok = wait_bar(cx, &full[slot], (n / S) & 1))) break;
          tc_fence_after_sync();
          const uint32_t sf = tmem + kTmemScaleBase + slot * 16;
          const uint8_t* asf = ASF + slot * 2 * kScaleAtomBytes;
          tc_copy_scales(sf + 0, desc_scales(asf));
          tc_copy_scales(sf + 4, desc_scales(asf + kScaleAtomBytes));
          tc_copy_scales(sf + 8, desc_scales(HSF + (hb * g.KC2 + c) * kScaleAtomBytes));
          const uint8_t* w = W + slot * kStageSmemWeights;
          const uint8_t* h = HC + (hb * g.KC2 + c) * kActImageBytes;
          const int ksteps = min(4, (g.I - c * kChunkK) / kBlock);
          for (int t = 0; t < 2; ++t)
            for (int kk = 0; kk < ksteps; ++kk)
              tc_mma_mxf8f6f4(tmem + set * 16 + t * 8,
                              desc_sw128(w + t * (kStageSmemWeights / 2) + kk * 32),
                              desc_sw128(h + kk * 32), mma_idesc(kk), sf + 4 * t, sf + 8,
                              (c == 0 && kk == 0) ? 0u : 1u);
          tc_commit(&empty[slot]);
          ++n;
        }
        if (!ok) break;
        meta[set] = make_int4(1, j, 0, 0);
        tc_commit(&accfull[set]);
        mbar_arrive(&accfull[set]);
        ++k;
      }
      // End marker for the epilogue (also after a timeout, so it exits).
      const int set = k % NACC;
      if (k >= NACC) wait_bar(cx, &accempty[set], ((k / NACC) - 1) & 1);
      meta[set] = make_int4(2, 0, 0, 0);
      mbar_arrive_count(&accfull[set], 2);
    }
  } else if (warp == 2) {
    // ------------------------------- activation gather (FC1), hidden loader (FC2)
    int n = 0, cu = -1;
    int tok_code = -1, tok_scale = -1;
    bool ok = true;
    for (int s = f0; s < f1 && ok; ++s) {
      const int item = s / g.KC1, c = s % g.KC1, u = item / g.P1;
      if (u != cu) {
        const int pc = a.unit_rows[u * kUnitRows + (lane >> 2)];
        const int ps = a.unit_rows[u * kUnitRows + (lane & 7)];
        tok_code = pc >= 0 ? (pc >> 4) : -1;
        tok_scale = ps >= 0 ? (ps >> 4) : -1;
        cu = u;
      }
      const int slot = n % S;
      if (n >= S) {
        bool freed = true;
        if (lane == 0) freed = wait_bar(cx, &empty[slot], ((n / S) & 1) ^ 1);
        if (!(ok = __shfl_sync(0xFFFFFFFFu, freed, 0))) break;
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
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // Hidden loader: one image per FC2 unit, double-buffered.
    int ordinal = -1;
    cu = -1;
    for (int j = j0; j < j1 && ok; ++j) {
      const int u = j / g.NQ;
      if (u == cu) continue;
      cu = u;
      ++ordinal;
      const int b = ordinal & 1;
      if (ordinal >= 2) {
        bool freed = true;
        if (lane == 0) freed = wait_bar(cx, &hempty[b], ((ordinal >> 1) - 1) & 1);
        if (!(ok = __shfl_sync(0xFFFFFFFFu, freed, 0))) break;
      }
      // Wait (bounded) for every K chunk of the unit's hidden vector.
      const uint64_t start = global_timer_ns();
      for (int c = 0; c < g.KC2; ++c) {
        const uint32_t* flag = a.hidden_flags + u * g.KC2 + c;
        for (uint32_t i = 0; load_acquire_gpu(flag) == 0; ++i) {
          if ((i & 15u) == 15u && global_timer_ns() - start > a.timeout_ns) {
            report(a.status, MOE_ERR_DEVICE_TIMEOUT);
            break;  // proceed with whatever the image holds
          }
        }
      }
      const uint8_t* src = a.hidden + static_cast<size_t>(u) * g.hidden_bytes;
      uint8_t* codes = HC + b * g.KC2 * kActImageBytes;
      uint8_t* scales = HSF + b * g.KC2 * kScaleAtomBytes;
      for (int i = lane; i < g.KC2 * kActImageBytes / 16; i += 32)
        reinterpret_cast<uint4*>(codes)[i] = load_cg_v4(src + i * 16);
      for (int i = lane; i < g.KC2 * kScaleAtomBytes / 16; i += 32)
        reinterpret_cast<uint4*>(scales)[i] = load_cg_v4(src + g.KC2 * kActImageBytes + i * 16);
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&hfull[b]);
    }
  } else if (warp >= kEpilogueWarp0) {
    // ------------------------------------------------------------ epilogue
    const int wq = warp - kEpilogueWarp0;  // TMEM lane quarter
    const int et = tid - kEpilogueWarp0 * 32;
    const int m = wq * 32 + lane;          // tile row of this thread
    int k = 0, out_unit = -1, out_pair = -1;
    for (;;) {
      const int set = k % NACC;
      if (!wait_bar(cx, &accfull[set], (k / NACC) & 1)) break;
      tc_fence_after_sync();
      const int4 md = meta[set];
      if (md.x == 2) break;
      float v0[8], v1[8];
      tmem_load_8(tmem + (static_cast<uint32_t>(wq * 32) << 16) + set * 16, v0);
      tmem_load_8(tmem + (static_cast<uint32_t>(wq * 32) << 16) + set * 16 + 8, v1);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[set]);
      ++k;
      if (md.x == 0) {
        // ---- FC1 piece: gate = v0, up = v1 for rows 128p + m.
        const int item = md.y, u = item / g.P1, p = item % g.P1;
        const uint4 rw = *reinterpret_cast<const uint4*>(a.unit_rows + u * kUnitRows);
        const int16_t* rows = reinterpret_cast<const int16_t*>(&rw);
        int valid = 0;
        while (valid < kUnitRows && rows[valid] >= 0) ++valid;
        const bool whole = (md.z % g.KC1 == 0) && (md.w % g.KC1 == g.KC1 - 1);
        if (!whole) {
          const int slot = (f0 >= item * g.KC1) ? 0 : 1;
          float* dst = a.partials + static_cast<size_t>(cta * 2 + slot) * 2 * kUnitRows * kTileM;
          for (int t = 0; t < valid; ++t) {
            dst[t * kTileM + m] = v0[t];
            dst[kUnitRows * kTileM + t * kTileM + m] = v1[t];
          }
          epilogue_sync();
          if (et == 0) {
            __threadfence();
            const uint32_t before = atomicAdd(&a.item_counters[item], 1u);
            const int c_lo = sp.cta_of(item * g.KC1), c_hi = sp.cta_of(item * g.KC1 + g.KC1 - 1);
            uint32_t pieces = 0;
            for (int c = c_lo; c <= c_hi; ++c) pieces += sp.fc1_begin(c) < sp.fc1_begin(c + 1);
            const bool last = before + 1 == pieces;
            if (last) __threadfence();
            misc[2] = last ? 1u : 0u;
          }
          epilogue_sync();
          const bool last = misc[2] != 0;
          epilogue_sync();  // misc[2] is reused by the next piece
          if (!last) continue;
          // Sum every piece in CTA order (deterministic whoever finishes last).
          float gs[8], us[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) gs[t] = us[t] = 0.f;
          const int c_lo = sp.cta_of(item * g.KC1), c_hi = sp.cta_of(item * g.KC1 + g.KC1 - 1);
          for (int c = c_lo; c <= c_hi; ++c) {
            const int b0 = sp.fc1_begin(c);
            if (b0 == sp.fc1_begin(c + 1)) continue;
            if (c == cta) {
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                gs[t] += v0[t];
                us[t] += v1[t];
              }
            } else {
              const int sl = (b0 >= item * g.KC1) ? 0 : 1;
              const float* src = a.partials + static_cast<size_t>(c * 2 + sl) * 2 * kUnitRows * kTileM;
              for (int t = 0; t < valid; ++t) {
                gs[t] += __ldcg(src + t * kTileM + m);
                us[t] += __ldcg(src + kUnitRows * kTileM + t * kTileM + m);
              }
            }
          }
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            v0[t] = gs[t];
            v1[t] = us[t];
          }
        }
        // SiLU(gate) * up, MXFP8 per 32 hidden values (= this warp's 32 rows).
        if (p * kTileM + wq * 32 < g.I) {
          uint8_t* img = a.hidden + static_cast<size_t>(u) * g.hidden_bytes;
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float h = t < valid ? silu_times(v0[t], v1[t]) : 0.f;
            float amax = fabsf(h);
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
            const int E = mx_exponent(amax, g.floor_rule != 0);
            img[p * kActImageBytes + swizzle128(t, m >> 4) + (m & 15)] = e4m3_code(h * pow2f(-E));
            if (lane == 0)
              img[g.KC2 * kActImageBytes + p * kScaleAtomBytes + scale_atom(t, wq)] =
                  static_cast<uint8_t>(E + 127);
          }
        }
        epilogue_sync();
        if (et == 0) {
          __threadfence();
          if (u != a.withhold_unit) store_release_gpu(&a.hidden_flags[u * g.KC2 + p], 1u);
        }
      } else {
        // ---- FC2 job: rows 256q + m (v0) and 256q + 128 + m (v1) -> BF16.
        const int j = md.y, u = j / g.NQ, q = j % g.NQ;
        if (u != out_unit) {
          out_pair = a.unit_rows[u * kUnitRows + (et >> 4)];
          out_unit = u;
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          OUT[t * 2 * kTileM + m] = __bfloat16_as_ushort(__float2bfloat16_rn(v0[t]));
          OUT[t * 2 * kTileM + kTileM + m] = __bfloat16_as_ushort(__float2bfloat16_rn(v1[t]));
        }
        epilogue_sync();
        if (out_pair >= 0) {
          const int r = et >> 4, ch = et & 15;
          uint16_t* dst = a.out + static_cast<size_t>(out_pair) * g.H + q * 2 * kTileM;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int chunk = ch + 16 * h;
            *reinterpret_cast<uint4*>(dst + chunk * 8) =
                *reinterpret_cast<const uint4*>(OUT + r * 2 * kTileM + chunk * 8);
          }
        }
        epilogue_sync();
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 3) tmem_dealloc(tmem, kTmemColumns);
}

}  // namespace

int experts_smem_bytes(const Geometry& g) { return Layout(g.KC2).bytes; }

cudaError_t experts_configure(const Geometry& g) {
  // The attribute belongs to the kernel, not to a handle: allow the largest
  // layout any handle can need (I = 512), so every prepared layer launches.
  (void)g;
  return cudaFuncSetAttribute(experts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Layout(kMaxInterChunks).bytes);
}

cudaError_t experts_occupancy(const Geometry& g, int* blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, experts_kernel, kThreads,
                                                       experts_smem_bytes(g));
}

cudaError_t launch_experts(const ExpertsArgs& a, int grid, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = experts_smem_bytes(a.g);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, experts_kernel, a);
}

}  // namespace moe
