// Routing-weighted combine (the single-GPU half of the pages' finalize step).
//
// Page: ...cutedsl.moe.experts, ExpertsKernel.finalize: every token's 16
// staged BF16 rows are summed with their routing weights, slot by slot, as
// FP32 multiply-adds, and the sum is stored once per token. Here the rows are
// the per-pair output of the run; pairs the grouping dropped (bad or
// repeated ids) wrote no row and are skipped. The result is rounded to BF16
// (nearest even).
//
// One thread per 8 consecutive outputs of a token: a 16-byte load of each
// slot's row (all issued together), eight FP32 accumulators, one 16-byte
// store. The kept flags and weights of a token are 16-byte aligned (the
// call checks the weights' alignment; the flags live in the workspace).
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kCombineThreads = 256;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineArgs a) {
  // No early trigger: the next call may read this call's output as its
  // input (stacked layers), before any wait of its own, so it starts only
  // once this grid has completed.
  ptx::grid_dependency_wait();  // the experts grid's rows
  const int per_token = a.H / 8;
  const int i = blockIdx.x * kCombineThreads + threadIdx.x;
  if (i >= a.B * per_token) return;
  const int t = i / per_token, n = (i - t * per_token) * 8;
  // Every load of the token's 16 slots is issued at once (one round trip):
  // the kept flags, the weights and the rows. A dropped pair's row is stale
  // and is never used: its slot is skipped, not multiplied by zero.
  const uint4 kept4 = __ldg(reinterpret_cast<const uint4*>(a.kept + t * kTopK));
  const float4* w4 = reinterpret_cast<const float4*>(a.weights + t * kTopK);
  float w[kTopK];
#pragma unroll
  for (int j = 0; j < kTopK / 4; ++j) {
    const float4 v = __ldg(w4 + j);
    w[4 * j] = v.x;
    w[4 * j + 1] = v.y;
    w[4 * j + 2] = v.z;
    w[4 * j + 3] = v.w;
  }
  uint4 row[kTopK];
#pragma unroll
  for (int s = 0; s < kTopK; ++s)
    row[s] = __ldg(reinterpret_cast<const uint4*>(a.rows + static_cast<size_t>(t * kTopK + s) * a.H + n));
  const uint32_t kept_words[4] = {kept4.x, kept4.y, kept4.z, kept4.w};
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.f;
#pragma unroll
  for (int s = 0; s < kTopK; ++s) {
    if (((kept_words[s >> 2] >> (8 * (s & 3))) & 0xFFu) == 0) continue;
    const uint32_t words[4] = {row[s].x, row[s].y, row[s].z, row[s].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc[2 * k] = fmaf(__uint_as_float(words[k] << 16), w[s], acc[2 * k]);
      acc[2 * k + 1] = fmaf(__uint_as_float(words[k] & 0xFFFF0000u), w[s], acc[2 * k + 1]);
    }
  }
  uint32_t packed[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    packed[k] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * k]))) |
                (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * k + 1]))) << 16);
  *reinterpret_cast<uint4*>(a.out + static_cast<size_t>(t) * a.H + n) =
      make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
  const int threads = a.B * (a.H / 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((threads + kCombineThreads - 1) / kCombineThreads);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.stream = stream;
  // Chained to the experts launch before it (programmatic dependent launch):
  // its blocks may be placed while that grid runs and wait for it to end.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

}  // namespace moe
