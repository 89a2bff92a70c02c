// One-time repack of caller weights (canonical row-major block format) into
// the tile format the expert kernels stream (layout described in common.cuh).
// Pure data movement: every code, scale and min is copied bit for bit.
#include "common.cuh"
#include "kernels.h"

namespace strata {

template <int BITS>
__global__ void repack_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scale,
                              const uint16_t* __restrict__ mn, int n, int rows, int K, uint8_t* __restrict__ out) {
  constexpr int kBlock = Fmt<BITS>::kBlock, kKstep = Fmt<BITS>::kKstep, kChunk = Fmt<BITS>::kChunk;
  const int nks = K / kKstep;
  const int nblk = K / kBlock;
  const int nmk = (nblk + 15) / 16;
  const int ntiles = rows / 16;
  const long long row_bytes = (long long)K * BITS / 8;
  const long long tile_bytes = (long long)nks * kChunk + nmk * 512;
  const long long per_tile = (long long)(nks + nmk) * 32;
  const long long total = (long long)n * ntiles * per_tile;
  for (long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x; item < total;
       item += (long long)gridDim.x * blockDim.x) {
    const int lane = (int)(item % 32);
    const long long rest = item / 32;
    const int j = (int)(rest % (nks + nmk));
    const long long mt = rest / (nks + nmk);  // matrix * ntiles + tile
    const int m = (int)(mt / ntiles), tile = (int)(mt % ntiles);
    const int g = lane >> 2, c = lane & 3;
    const uint8_t* cm = codes + (long long)m * rows * row_bytes;
    const uint16_t* sm = scale + (long long)m * rows * nblk;
    const uint16_t* mm = mn + (long long)m * rows * nblk;
    uint8_t* tb = out + mt * tile_bytes;
    const int rg = tile * 16 + g, r8 = rg + 8;
    if (j < nks) {
      const int ks = j;
      uint32_t words[4];
      if (BITS == 4) {
        // word (row, block): lane c's elements 8c..8c+7, element u at bit
        // (u odd ? 16 : 0) + 4*(u/2)
        for (int wi = 0; wi < 4; ++wi) {
          const int row = (wi & 1) ? r8 : rg;
          const int beta = 2 * ks + (wi >> 1);
          const uint8_t* src = cm + (long long)row * row_bytes + beta * 16 + 4 * c;
          uint32_t cw = (uint32_t)src[0] | ((uint32_t)src[1] << 8) | ((uint32_t)src[2] << 16) | ((uint32_t)src[3] << 24);
          uint32_t w = 0;
          for (int u = 0; u < 8; ++u) w |= ((cw >> (4 * u)) & 15u) << (((u & 1) ? 16 : 0) + 4 * (u >> 1));
          words[wi] = w;
        }
      } else {
        // word wi covers blocks (2wi, 2wi+1) of the k-step for rows g and g+8;
        // pair p = rowsel*4 + bsel*2 + (u/2) at bits (2p, 2p+16)
        for (int wi = 0; wi < 4; ++wi) {
          uint32_t w = 0;
          for (int rowsel = 0; rowsel < 2; ++rowsel) {
            const int row = rowsel ? r8 : rg;
            for (int bsel = 0; bsel < 2; ++bsel) {
              const int beta = 8 * ks + 2 * wi + bsel;
              const uint32_t byte = cm[(long long)row * row_bytes + beta * 4 + c];
              for (int u = 0; u < 4; ++u) {
                const uint32_t q = (byte >> (2 * u)) & 3u;
                const int p = rowsel * 4 + bsel * 2 + (u >> 1);
                w |= q << (2 * p + 16 * (u & 1));
              }
            }
          }
          words[wi] = w;
        }
      }
      uint8_t* ch = tb + (long long)ks * kChunk;
      *reinterpret_cast<uint4*>(ch + lane * 16) = make_uint4(words[0], words[1], words[2], words[3]);
      if (c == 0) {
        uint16_t* rec = reinterpret_cast<uint16_t*>(ch + 512 + g * Fmt<BITS>::kScaleRec);
        if (BITS == 4) {
          rec[0] = sm[(long long)rg * nblk + 2 * ks];
          rec[1] = sm[(long long)rg * nblk + 2 * ks + 1];
          rec[2] = sm[(long long)r8 * nblk + 2 * ks];
          rec[3] = sm[(long long)r8 * nblk + 2 * ks + 1];
        } else {
          for (int b = 0; b < 8; ++b) {
            rec[b] = sm[(long long)rg * nblk + 8 * ks + b];
            rec[8 + b] = sm[(long long)r8 * nblk + 8 * ks + b];
          }
        }
      }
    } else {
      const int mk = j - nks;
      const int b0 = mk * 16 + 2 * c, b8 = b0 + 8;
      auto mv = [&](int row, int beta) -> uint16_t { return beta < nblk ? mm[(long long)row * nblk + beta] : 0; };
      uint16_t* dst = reinterpret_cast<uint16_t*>(tb + (long long)nks * kChunk + mk * 512 + lane * 16);
      dst[0] = mv(rg, b0);
      dst[1] = mv(rg, b0 + 1);
      dst[2] = mv(r8, b0);
      dst[3] = mv(r8, b0 + 1);
      dst[4] = mv(rg, b8);
      dst[5] = mv(rg, b8 + 1);
      dst[6] = mv(r8, b8);
      dst[7] = mv(r8, b8 + 1);
    }
  }
}

long long packed_bytes(int n, int rows, int K, int bits) {
  const int kstep = bits == 4 ? 64 : 128, block = bits == 4 ? 32 : 16, chunk = bits == 4 ? 576 : 768;
  const long long tile = (long long)(K / kstep) * chunk + (long long)((K / block + 15) / 16) * 512;
  return (long long)n * (rows / 16) * tile;
}

PackedMat packed_desc(const uint8_t* base, int rows, int K, int bits) {
  PackedMat M;
  const int kstep = bits == 4 ? 64 : 128, block = bits == 4 ? 32 : 16, chunk = bits == 4 ? 576 : 768;
  M.base = base;
  M.rows = rows;
  M.K = K;
  M.nks = K / kstep;
  M.nmk = (K / block + 15) / 16;
  M.tile_bytes = M.nks * chunk + M.nmk * 512;
  M.mat_bytes = (long long)(rows / 16) * M.tile_bytes;
  return M;
}

cudaError_t launch_repack(const uint8_t* codes, const uint16_t* scale, const uint16_t* mn, int n, int rows, int K,
                          int bits, uint8_t* out, cudaStream_t s) {
  const int kstep = bits == 4 ? 64 : 128, block = bits == 4 ? 32 : 16;
  const long long items = (long long)n * (rows / 16) * (K / kstep + (K / block + 15) / 16) * 32;
  long long blocks = (items + 255) / 256;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  if (bits == 4) repack_kernel<4><<<(unsigned)blocks, 256, 0, s>>>(codes, scale, mn, n, rows, K, out);
  else repack_kernel<2><<<(unsigned)blocks, 256, 0, s>>>(codes, scale, mn, n, rows, K, out);
  return cudaGetLastError();
}

}  // namespace strata
