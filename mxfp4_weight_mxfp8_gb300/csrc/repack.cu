// Weight repack (moe_prepare): the caller's row-major MXFP4 arrays become one
// contiguous 17,408-byte block per weight stage, in the order the persistent
// experts kernel streams them, so every TMA stage is a single linear read.
//
// Stage block: [tile 0: 128 rows x 64 B][tile 1: 128 rows x 64 B]
//              [tile 0 scale atom 512 B][tile 1 scale atom 512 B]
// FC1 stage (pair p, K chunk c): tile 0 = gate rows 128p .. 128p+127,
//   tile 1 = the matching up rows I + 128p ..; rows past I are zero.
// FC2 stage (tile pair q, K chunk c): tiles = output rows 256q .. 256q+127
//   and 256q+128 .. 256q+255; K columns past I are zero.
// Scale atoms hold (row r, k-block kb) at (r % 32) * 16 + (r / 32) * 4 + kb,
// the layout of the tensor core's 32x128b scale-factor copy.
#include "kernels.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) repack_kernel(const uint8_t* __restrict__ w13,
                                                     const uint8_t* __restrict__ s13,
                                                     const uint8_t* __restrict__ w2,
                                                     const uint8_t* __restrict__ s2,
                                                     const Geometry g, uint8_t* __restrict__ stages) {
  const int block = blockIdx.x;
  const int e = block / g.SPE, s = block % g.SPE;
  const int t = threadIdx.x >> 7, r = threadIdx.x & 127;  // tile, row within tile
  uint8_t* dst = stages + static_cast<size_t>(block) * kStageBytes;
  uint8_t* dw = dst + t * kTileBytes + r * (kChunkK / 2);
  uint8_t* ds = dst + kStageWeightBytes + t * kScaleAtomBytes;
  const uint8_t* src_w = nullptr;
  const uint8_t* src_s = nullptr;
  int valid_bytes = 0, valid_blocks = 0;
  if (s < g.P1 * g.KC1) {
    const int p = s / g.KC1, c = s % g.KC1;
    const int j = p * kTileM + r;
    if (j < g.I) {
      const size_t row = static_cast<size_t>(e) * 2 * g.I + (t == 0 ? 0 : g.I) + j;
      src_w = w13 + row * (g.H / 2) + c * (kChunkK / 2);
      src_s = s13 + row * (g.H / kBlock) + c * (kChunkK / kBlock);
      valid_bytes = kChunkK / 2;
      valid_blocks = kChunkK / kBlock;
    }
  } else {
    const int f = s - g.P1 * g.KC1, q = f / g.KC2, c = f % g.KC2;
    const size_t row = static_cast<size_t>(e) * g.H + q * 2 * kTileM + t * kTileM + r;
    const int k0 = c * kChunkK, kvalid = min(kChunkK, g.I - k0);
    src_w = w2 + row * (g.I / 2) + k0 / 2;
    src_s = s2 + row * (g.I / kBlock) + k0 / kBlock;
    valid_bytes = kvalid / 2;
    valid_blocks = kvalid / kBlock;
  }
  for (int b = 0; b < kChunkK / 2; b += 16) {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (b < valid_bytes) v = *reinterpret_cast<const uint4*>(src_w + b);  // valid_bytes % 16 == 0
    *reinterpret_cast<uint4*>(dw + b) = v;
  }
  for (int kb = 0; kb < kChunkK / kBlock; ++kb)
    ds[scale_atom(r, kb)] = kb < valid_blocks ? src_s[kb] : 0;
}

}  // namespace

cudaError_t launch_repack(const uint8_t* w13, const uint8_t* s13, const uint8_t* w2,
                          const uint8_t* s2, const Geometry& g, uint8_t* stages,
                          cudaStream_t stream) {
  const int blocks = g.E * g.SPE;
  repack_kernel<<<blocks, 256, 0, stream>>>(w13, s13, w2, s2, g, stages);
  return cudaGetLastError();
}

}  // namespace moe
