// q4k_pack: Q4_K fields -> 144-byte superblocks (GGUF Q4_K byte order), and
// its inverse q4k_unpack (a test export: superblocks -> fields).
//
// One warp packs one superblock: lane l writes quant bytes 4l..4l+3 (the
// 64-weight chunk c = l/8 pairs weight 64c+i in the low nibble with weight
// 64c+32+i in the high nibble), lanes 0..3 write the 16 header bytes.  All
// global accesses are 4-byte words, coalesced within the warp.  Unpacking
// reads the same words and writes the fields back the same way.
#include "q4k_internal.h"

namespace q4k {
namespace {

__device__ __forceinline__ uint32_t byte_of(uint32_t v, int i) { return (v >> (8 * i)) & 0xFFu; }

__global__ void __launch_bounds__(256) pack_block144_kernel(
    const uint16_t* __restrict__ d, const uint16_t* __restrict__ dmin,
    const uint8_t* __restrict__ sc, const uint8_t* __restrict__ m,
    const uint8_t* __restrict__ q, int64_t n_super, int64_t nb,
    uint8_t* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t sb = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       sb < n_super; sb += warps_total) {
    const int64_t row = sb / nb;
    const int64_t col0 = (sb - row * nb) * kQK;
    const int64_t cols = nb * kQK;
    uint32_t* out = reinterpret_cast<uint32_t*>(w + sb * kBlockBytes);
    // quant bytes: lane l covers bytes 4l..4l+3 of the 128 quant bytes
    const int c = lane >> 3;
    const int i0 = (lane & 7) * 4;
    const uint8_t* qrow = q + row * cols + col0 + 64 * c + i0;
    const uint32_t lo = *reinterpret_cast<const uint32_t*>(qrow) & 0x0F0F0F0Fu;
    const uint32_t hi = *reinterpret_cast<const uint32_t*>(qrow + 32) & 0x0F0F0F0Fu;
    out[4 + lane] = lo | (hi << 4);
    if (lane < 4) {
      uint32_t word;
      if (lane == 0) {
        word = (uint32_t)d[sb] | ((uint32_t)dmin[sb] << 16);
      } else {
        const uint8_t* scp = sc + row * (cols / kSub) + (col0 / kSub);
        const uint8_t* mp = m + row * (cols / kSub) + (col0 / kSub);
        const uint32_t s_lo = *reinterpret_cast<const uint32_t*>(scp) & 0x3F3F3F3Fu;
        const uint32_t s_hi = *reinterpret_cast<const uint32_t*>(scp + 4) & 0x3F3F3F3Fu;
        const uint32_t m_lo = *reinterpret_cast<const uint32_t*>(mp) & 0x3F3F3F3Fu;
        const uint32_t m_hi = *reinterpret_cast<const uint32_t*>(mp + 4) & 0x3F3F3F3Fu;
        word = 0;
        for (int j = 0; j < 4; ++j) {
          uint32_t b;
          if (lane == 1) {        // scale bytes 0..3: sc_j | (sc_{j+4} >> 4) << 6
            b = byte_of(s_lo, j) | ((byte_of(s_hi, j) >> 4) << 6);
          } else if (lane == 2) { // scale bytes 4..7: m_j | (m_{j+4} >> 4) << 6
            b = byte_of(m_lo, j) | ((byte_of(m_hi, j) >> 4) << 6);
          } else {                // scale bytes 8..11: low nibbles of sc_{j+4}, m_{j+4}
            b = (byte_of(s_hi, j) & 15u) | ((byte_of(m_hi, j) & 15u) << 4);
          }
          word |= b << (8 * j);
        }
      }
      out[lane] = word;
    }
  }
}

// Inverse of pack_block144_kernel: one warp per superblock; lane l reads
// quant word l and writes its low nibbles to weights 64c+i and its high
// nibbles to 64c+32+i; lane 0 writes d and dmin, lanes 0..7 the sc and m of
// sub-block l.
__global__ void __launch_bounds__(256) unpack_block144_kernel(
    const uint8_t* __restrict__ w, int64_t n_super, int64_t nb, uint16_t* __restrict__ d,
    uint16_t* __restrict__ dmin, uint8_t* __restrict__ sc, uint8_t* __restrict__ m,
    uint8_t* __restrict__ q) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t sb = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       sb < n_super; sb += warps_total) {
    const int64_t row = sb / nb;
    const int64_t col0 = (sb - row * nb) * kQK;
    const int64_t cols = nb * kQK;
    const uint32_t* in = reinterpret_cast<const uint32_t*>(w + sb * kBlockBytes);
    const uint32_t word = in[4 + lane];
    const int c = lane >> 3;
    const int i0 = (lane & 7) * 4;
    uint8_t* qrow = q + row * cols + col0 + 64 * c + i0;
    *reinterpret_cast<uint32_t*>(qrow) = word & 0x0F0F0F0Fu;
    *reinterpret_cast<uint32_t*>(qrow + 32) = (word >> 4) & 0x0F0F0F0Fu;
    if (lane == 0) {
      const uint32_t h = in[0];
      d[sb] = (uint16_t)(h & 0xFFFFu);
      dmin[sb] = (uint16_t)(h >> 16);
    }
    if (lane < 8) {
      const uint32_t s03 = in[1], m03 = in[2], x47 = in[3];
      const int j = lane;
      uint32_t scj, mj;
      if (j < 4) {
        scj = byte_of(s03, j) & 63u;
        mj = byte_of(m03, j) & 63u;
      } else {
        scj = (byte_of(x47, j - 4) & 15u) | ((byte_of(s03, j - 4) >> 6) << 4);
        mj = (byte_of(x47, j - 4) >> 4) | ((byte_of(m03, j - 4) >> 6) << 4);
      }
      const int64_t sub = row * (cols / kSub) + col0 / kSub + j;
      sc[sub] = (uint8_t)scj;
      m[sub] = (uint8_t)mj;
    }
  }
}

int pack_grid(int64_t n_super) {
  int dev = 0;
  cudaGetDevice(&dev);
  const int64_t want = (n_super + 7) / 8;
  const int64_t cap = (int64_t)device_info(dev).sm_count * 16;
  return (int)(want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_unpack_block144(const uint8_t* w, int64_t rows, int64_t cols, uint16_t* d, uint16_t* dmin,
                                   uint8_t* sc, uint8_t* m, uint8_t* q, cudaStream_t s) {
  const int64_t nb = cols / kQK;
  const int64_t n_super = rows * nb;
  if (n_super == 0) return cudaSuccess;
  unpack_block144_kernel<<<pack_grid(n_super), 256, 0, s>>>(w, n_super, nb, d, dmin, sc, m, q);
  return cudaGetLastError();
}

cudaError_t launch_pack_block144(const uint16_t* d, const uint16_t* dmin,
                                 const uint8_t* sc, const uint8_t* m,
                                 const uint8_t* q, int64_t rows, int64_t cols,
                                 uint8_t* w, cudaStream_t s) {
  const int64_t nb = cols / kQK;
  const int64_t n_super = rows * nb;
  if (n_super == 0) return cudaSuccess;
  pack_block144_kernel<<<pack_grid(n_super), 256, 0, s>>>(d, dmin, sc, m, q, n_super, nb, w);
  return cudaGetLastError();
}

}  // namespace q4k
