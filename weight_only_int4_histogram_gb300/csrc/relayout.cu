// Plan-time relayout of packed INT4 expert weights into the interleaved,
// K-packed layout the GEMM kernels dequantise without byte permutes.
//
// "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy), section
// Motivation (weights stay packed INT4; no persistent BF16 expansion) and
// "[None][feat] Add W4A16 per-channel weight-only support for Cutlass fused
// MoE" (TensorRT-LLM), section Changes (a setup-time preprocessing of the
// packed weights for the mixed-input GEMM): the same bytes, reordered once
// before any forward.  The order is this library's own, chosen for the
// Blackwell dequantisation in gemm.cuh / gemv.cuh:
//
//   output [E, N, K/2] bytes, rows packed along K; in every 32-bit word w of a
//   row (K values 8w .. 8w + 7) the nibble at bit position 4p holds the code
//   of K index 8w + {0, 2, 4, 6, 1, 3, 5, 7}[p], so (word >> 4i) & 0x000F000F
//   is the pair (8w + 2i, 8w + 2i + 1) in the two 16-bit halves.
//
// Inputs are the checkpoint layouts of the C ABI: group scales [E, N, K/2]
// (byte b of a row = K 2b low | K 2b+1 high) or per-channel [E, N/2, K]
// (byte [p, k] = row 2p low | row 2p+1 high).  Codes are copied bit for bit.
#include "common.cuh"

namespace w4a16 {

// K-packed checkpoint word -> interleaved word (nibble position p of the input
// holds K index p).
__device__ __forceinline__ uint32_t interleave_word(uint32_t x) {
  uint32_t y = 0;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int k = (p < 4) ? 2 * p : 2 * (p - 4) + 1;  // K index stored at output position p
    y |= ((x >> (4 * k)) & 0xFu) << (4 * p);
  }
  return y;
}

// One thread per 32-bit word; in == out is allowed (each word maps to itself).
__global__ void __launch_bounds__(256) relayout_kpacked_kernel(const uint32_t* in, uint32_t* out, int64_t n_words) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_words; i += stride)
    out[i] = interleave_word(in[i]);
}

// Row-pair packed [E, N/2, K] -> interleaved K-packed [E, N, K/2]: one thread
// per output word (row n, K values 8w .. 8w + 7), reading the 8 bytes of row
// pair n / 2 at those K and taking nibble n % 2 of each.
__global__ void __launch_bounds__(256) relayout_rowpair_kernel(const uint8_t* in, uint32_t* out, int64_t E, int32_t N,
                                                               int32_t K) {
  const int32_t words_row = K / 8;
  const int64_t n_words = E * N * static_cast<int64_t>(words_row);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_words; i += stride) {
    const int64_t row = i / words_row;  // e * N + n
    const int32_t w = static_cast<int32_t>(i - row * words_row);
    const int64_t e = row / N;
    const int32_t n = static_cast<int32_t>(row - e * N);
    const uint2 b = *reinterpret_cast<const uint2*>(in + (e * (N / 2) + n / 2) * static_cast<int64_t>(K) + 8 * w);
    const int sh = (n & 1) * 4;
    uint32_t x = 0;  // K-packed checkpoint word of row n: nibble position j = K 8w + j
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x |= ((b.x >> (8 * j + sh)) & 0xFu) << (4 * j);
      x |= ((b.y >> (8 * j + sh)) & 0xFu) << (4 * (j + 4));
    }
    out[i] = interleave_word(x);
  }
}

cudaError_t launch_relayout(bool row_pairs, const uint8_t* in, uint8_t* out, int64_t E, int32_t N, int32_t K,
                            int num_sms, cudaStream_t s) {
  const int64_t n_words = E * N * static_cast<int64_t>(K / 8);
  const int64_t blocks = (n_words + 255) / 256;
  const unsigned grid = static_cast<unsigned>(blocks < 8LL * num_sms ? (blocks > 0 ? blocks : 1) : 8LL * num_sms);
  if (row_pairs)
    relayout_rowpair_kernel<<<grid, 256, 0, s>>>(in, reinterpret_cast<uint32_t*>(out), E, N, K);
  else
    relayout_kpacked_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint32_t*>(in),
                                                 reinterpret_cast<uint32_t*>(out), n_words);
  return cudaGetLastError();
}

}  // namespace w4a16
