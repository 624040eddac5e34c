// Q6_K weights: conversions between the fields (d, sc, q), the 210-byte GGUF
// superblocks and the GPU row layout the decode GEMV streams with tensor
// copies (genie-ai-runtime §6, Path G: a Q6_K block layout redesigned for
// vectorised loads).
//
// GGUF superblock (210 bytes, 256 weights): ql[128] low 4 bits, qh[64] high
// 2 bits, 16 int8 scales (one per 16 weights), binary16 d; w = d*sc*(q - 32).
// Within half n (weights 128n..128n+127) and l < 32: ql[64n+l] holds weights
// 128n+l (low nibble) and 128n+64+l (high), ql[64n+32+l] weights 128n+32+l
// and 128n+96+l, and qh[32n+l] the high bits of 128n+l, +32+l, +64+l, +96+l
// in bit pairs 0-1, 2-3, 4-5, 6-7.
//
// GPU layout (q6k_gpu_row_bytes per row, rows back to back): the row's nb
// superblocks of 208 bytes, then the nb values of d (binary16), then zero
// padding to a multiple of 16 bytes.  A superblock: the 16 int8 scales, then
// four 48-byte chunks of 64 weights.  Chunk c covers weights 64c..64c+63, as
// sub-block s = 0 (64c..64c+31) and s = 1 (64c+32..64c+63):
//  - bytes 0..31: byte t holds the low 4 bits of weight 64c+t (low nibble)
//    and of 64c+32+t (high nibble);
//  - bytes 32..47: byte i holds, in bit pair 2f (f = 2s + h), the high 2 bits
//    of weight 64c + 32s + 16h + i, with the upper bit of the pair inverted.
// So every superblock starts on a 16-byte boundary, a row is one tensor copy
// of 208-byte boxes plus one of d, and the GEMV assembles a signed byte
// 4*(q - 32) from one low nibble and one bit pair with a shift and a mask each
// (the inverted bit makes the pair the byte's sign bits).
//
// Conversion kernels run one warp per superblock: the warp gathers the
// superblock's 256 quants, 16 scales and d into shared memory, then writes
// the output bytes with consecutive lanes on consecutive bytes.
#include "q4k_internal.h"

namespace q4k {
namespace {

constexpr int kWarps = 8;

struct Q6Smem {
  uint8_t q[kQK];
  int8_t sc[16];
  uint16_t d;
};

// quant of weight pos (0..255) of a GGUF superblock
__device__ __forceinline__ uint32_t gguf_q(const uint8_t* b, int pos) {
  const int n = pos >> 7, r = pos & 127, quarter = r >> 5, l = r & 31;
  const uint32_t lo = (b[64 * n + 32 * (quarter & 1) + l] >> (4 * (quarter >> 1))) & 15u;
  const uint32_t hi = (b[128 + 32 * n + l] >> (2 * quarter)) & 3u;
  return lo | (hi << 4);
}

// quant of weight pos (0..255) of a GPU superblock
__device__ __forceinline__ uint32_t gpu_q(const uint8_t* b, int pos) {
  const int c = pos >> 6, s = (pos >> 5) & 1, t = pos & 31, h = t >> 4;
  const uint8_t* ch = b + 16 + 48 * c;
  const uint32_t lo = (ch[t] >> (4 * s)) & 15u;
  const uint32_t hi = ((ch[32 + (t & 15)] >> (2 * (2 * s + h))) & 3u) ^ 2u;
  return lo | (hi << 4);
}

// byte i (0..209) of the GGUF superblock of S
__device__ __forceinline__ uint8_t gguf_byte(const Q6Smem& S, int i) {
  if (i < 128) {
    const int n = i >> 6, l = i & 63;
    return (uint8_t)((S.q[128 * n + l] & 15u) | ((S.q[128 * n + 64 + l] & 15u) << 4));
  }
  if (i < 192) {
    const int j = i - 128, n = j >> 5, l = j & 31;
    const uint8_t* q = S.q + 128 * n + l;
    return (uint8_t)((q[0] >> 4) | ((q[32] >> 4) << 2) | ((q[64] >> 4) << 4) | ((q[96] >> 4) << 6));
  }
  if (i < 208) return (uint8_t)S.sc[i - 192];
  return i == 208 ? (uint8_t)(S.d & 0xFFu) : (uint8_t)(S.d >> 8);
}

// byte i (0..207) of the GPU superblock of S
__device__ __forceinline__ uint8_t gpu_byte(const Q6Smem& S, int i) {
  if (i < 16) return (uint8_t)S.sc[i];
  const int j = i - 16, c = j / 48, r = j - 48 * c;
  const uint8_t* q = S.q + 64 * c;
  if (r < 32) return (uint8_t)((q[r] & 15u) | ((q[32 + r] & 15u) << 4));
  const int t = r - 32;
  uint32_t v = 0;
#pragma unroll
  for (int f = 0; f < 4; ++f) v |= (((uint32_t)(q[32 * (f >> 1) + 16 * (f & 1) + t] >> 4) ^ 2u) & 3u) << (2 * f);
  return (uint8_t)v;
}

struct Q6Io {
  // fields (either side)
  const uint16_t* d_in;
  const int8_t* sc_in;
  const uint8_t* q_in;
  uint16_t* d_out;
  int8_t* sc_out;
  uint8_t* q_out;
  // packed weights
  const uint8_t* w_in;
  uint8_t* w_out;
  int in_layout;     // -1 fields, Q6K_LAYOUT_GGUF (0) or Q6K_LAYOUT_GPU (1)
  int out_layout;
  int64_t n_super, nb, row_bytes;
};

__global__ void __launch_bounds__(32 * kWarps) q6k_convert_kernel(const Q6Io io) {
  __shared__ Q6Smem sm[kWarps];
  __shared__ __align__(16) uint8_t raw[kWarps][224];
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  Q6Smem& S = sm[wi];
  uint8_t* R = raw[wi];
  const int64_t warps_total = (int64_t)gridDim.x * kWarps;
  for (int64_t sb = (int64_t)blockIdx.x * kWarps + wi; sb < io.n_super; sb += warps_total) {
    const int64_t row = sb / io.nb, blk = sb - row * io.nb;
    const int64_t cols = io.nb * kQK;
    // ---- gather the superblock
    if (io.in_layout < 0) {
      const uint8_t* q = io.q_in + row * cols + blk * kQK;
#pragma unroll
      for (int i = 0; i < 8; ++i) S.q[lane + 32 * i] = q[lane + 32 * i] & 63u;
      if (lane < 16) S.sc[lane] = io.sc_in[row * (cols / 16) + blk * 16 + lane];
      if (lane == 0) S.d = io.d_in[sb];
      __syncwarp();
    } else {
      const bool gguf = io.in_layout == 0;
      const uint8_t* src = gguf ? io.w_in + sb * kQ6GgufBytes : io.w_in + row * io.row_bytes + blk * kQ6GpuBytes;
      const int n = gguf ? kQ6GgufBytes : kQ6GpuBytes;
      for (int i = lane; i < n; i += 32) R[i] = src[i];
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int pos = lane + 32 * i;
        S.q[pos] = (uint8_t)(gguf ? gguf_q(R, pos) : gpu_q(R, pos));
      }
      if (lane < 16) S.sc[lane] = (int8_t)R[gguf ? 192 + lane : lane];
      if (lane == 0) {
        if (gguf) S.d = (uint16_t)(R[208] | (R[209] << 8));
        else S.d = *reinterpret_cast<const uint16_t*>(io.w_in + row * io.row_bytes + io.nb * kQ6GpuBytes + 2 * blk);
      }
      __syncwarp();
    }
    // ---- write it
    if (io.out_layout < 0) {
      uint8_t* q = io.q_out + row * cols + blk * kQK;
#pragma unroll
      for (int i = 0; i < 8; ++i) q[lane + 32 * i] = S.q[lane + 32 * i];
      if (lane < 16) io.sc_out[row * (cols / 16) + blk * 16 + lane] = S.sc[lane];
      if (lane == 0) io.d_out[sb] = S.d;
    } else if (io.out_layout == 0) {
      uint8_t* dst = io.w_out + sb * kQ6GgufBytes;
      for (int i = lane; i < kQ6GgufBytes; i += 32) dst[i] = gguf_byte(S, i);
    } else {
      uint8_t* rowp = io.w_out + row * io.row_bytes;
      uint8_t* dst = rowp + blk * kQ6GpuBytes;
      for (int i = lane; i < kQ6GpuBytes; i += 32) dst[i] = gpu_byte(S, i);
      if (lane == 0) *reinterpret_cast<uint16_t*>(rowp + io.nb * kQ6GpuBytes + 2 * blk) = S.d;
      // the row's zero padding, written with its last superblock
      const int64_t pad0 = io.nb * kQ6GgufBytes;
      if (blk == io.nb - 1 && pad0 + lane < io.row_bytes) rowp[pad0 + lane] = 0;
    }
    __syncwarp();
  }
}

}  // namespace

int64_t q6k_gpu_row_bytes(int64_t nb) { return (nb * kQ6GgufBytes + 15) / 16 * 16; }

cudaError_t launch_q6k_convert(const uint16_t* d_in, const int8_t* sc_in, const uint8_t* q_in, const uint8_t* w_in,
                               int in_layout, int64_t rows, int64_t cols, uint16_t* d_out, int8_t* sc_out,
                               uint8_t* q_out, uint8_t* w_out, int out_layout, cudaStream_t s) {
  Q6Io io{};
  io.d_in = d_in;
  io.sc_in = sc_in;
  io.q_in = q_in;
  io.w_in = w_in;
  io.d_out = d_out;
  io.sc_out = sc_out;
  io.q_out = q_out;
  io.w_out = w_out;
  io.in_layout = in_layout;
  io.out_layout = out_layout;
  io.nb = cols / kQK;
  io.n_super = rows * io.nb;
  io.row_bytes = q6k_gpu_row_bytes(io.nb);
  if (io.n_super == 0) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  const int64_t want = (io.n_super + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)device_info(dev).sm_count * 8;
  q6k_convert_kernel<<<(unsigned)(want < cap ? want : cap), 32 * kWarps, 0, s>>>(io);
  return cudaGetLastError();
}

}  // namespace q4k
