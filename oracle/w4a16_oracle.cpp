// Plain, slow CPU oracle for the local W4A16 MoE forward.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
// baseline leg of the benchmark load this file's library; the product path
// never does, and this file shares no code, header or table with the CUDA
// kernels.  Parity pins for every function live in tests/test_oracle_pins.py.
//
// What it follows (each step restated from the pages, in their order):
//   * "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy), sections
//     *Modification* and *Benchmark*: routes -> gate/up GEMM -> SiLU ->
//     down GEMM -> weighted reduction; INT4 group size 32 with BF16 scales;
//     invalid routes and masked expert counts.
//   * "perf: reduce split W4A16 routing and output overhead" (FlashInfer),
//     section *Description*: per-expert outputs are combined in FP32 in fixed
//     top-k order, followed by one cast to the output dtype.
//   * "[None][feat] Add W4A16 per-channel weight-only support for Cutlass
//     fused MoE" (TensorRT-LLM), sections *Checkpoint format* (per-channel
//     packing along the output dim, even index in the low nibble) and
//     *Validation* (non-gated Relu2 arm).
//
// Precision: dequantisation, both expert GEMMs and the activation are done in
// double (the exact reading of the math); each route's expert output is then
// stored as FP32 and the combine is FP32, j ascending, exactly as the pages
// fix it.  Compiled with -ffp-contract=off so every float operation below is
// rounded as written.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ---------------------------------------------------------------------------
// 16-bit float formats (IEEE binary16 and bfloat16), decoded from their
// definitions and encoded with round-to-nearest-even.
// ---------------------------------------------------------------------------
double bf16_decode(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

double fp16_decode(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int ex = (h >> 10) & 0x1F;
  const int man = h & 0x3FF;
  double v;
  if (ex == 0) {
    v = std::ldexp(static_cast<double>(man), -24);
  } else if (ex == 31) {
    v = man ? NAN : INFINITY;
  } else {
    v = std::ldexp(1.0 + man / 1024.0, ex - 15);
  }
  return sign ? -v : v;
}

uint16_t bf16_encode(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;  // NaN
  u += 0x7FFFu + ((u >> 16) & 1u);                     // nearest, ties to even
  return static_cast<uint16_t>(u >> 16);
}

uint16_t fp16_encode(float f) {
  const double x = static_cast<double>(f);
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  const double a = std::fabs(x);
  if (std::isnan(x)) return 0x7E00;
  if (a == 0.0) return sign;
  int e2;
  std::frexp(a, &e2);          // a in [2^(e2-1), 2^e2)
  int E = e2 - 1;
  const double quantum = (E < -14) ? std::ldexp(1.0, -24) : std::ldexp(1.0, E - 10);
  const double r = std::nearbyint(a / quantum);  // default rounding: ties to even
  const double v = r * quantum;
  if (v >= 65536.0 || (v > 65504.0)) return sign | 0x7C00;  // overflow -> inf
  if (v < std::ldexp(1.0, -14)) {
    return sign | static_cast<uint16_t>(r);  // subnormal (r == 1024 is the min normal)
  }
  std::frexp(v, &e2);
  E = e2 - 1;
  const int man = static_cast<int>((v / std::ldexp(1.0, E) - 1.0) * 1024.0);
  return sign | static_cast<uint16_t>(((E + 15) << 10) | man);
}

// Signed INT4 code of a nibble: two's complement, range [-8, 7].
int int4_value(unsigned nibble) {
  nibble &= 0xFu;
  return nibble < 8 ? static_cast<int>(nibble) : static_cast<int>(nibble) - 16;
}

struct Desc {
  int32_t num_experts, expert_offset, hidden, inter, top_k, act, scale_kind, act_dtype;
};

int local_expert(const Desc& d, int32_t id) {
  if (id == -1) return -1;
  const int64_t l = static_cast<int64_t>(id) - d.expert_offset;
  return (l >= 0 && l < d.num_experts) ? static_cast<int>(l) : -1;
}

// Dequantised weight matrix of one expert, rows x cols (row = output channel,
// col = reduction index), in double.  group mode: packed [rows, cols/2] along
// cols with scales [rows, cols/32]; per-channel: packed [rows/2, cols] along
// rows with scales [rows].
void dequant_matrix(const uint8_t* packed, const uint16_t* scales, int64_t rows, int64_t cols,
                    int scale_kind, double* out) {
  for (int64_t n = 0; n < rows; ++n) {
    for (int64_t k = 0; k < cols; ++k) {
      int q;
      double s;
      if (scale_kind == 0) {
        const uint8_t byte = packed[n * (cols / 2) + k / 2];
        q = int4_value((k % 2 == 0) ? byte : (byte >> 4));
        s = bf16_decode(scales[n * (cols / 32) + k / 32]);
      } else {
        const uint8_t byte = packed[(n / 2) * cols + k];
        q = int4_value((n % 2 == 0) ? byte : (byte >> 4));
        s = bf16_decode(scales[n]);
      }
      out[n * cols + k] = static_cast<double>(q) * s;
    }
  }
}

double silu(double g) { return g / (1.0 + std::exp(-g)); }

}  // namespace

extern "C" {

int oracle_abi_version(void) { return 1; }

// Nibble unpacking, exposed for the packing pins.
void oracle_unpack_along_k(const uint8_t* packed, int64_t rows, int64_t cols, int8_t* q) {
  for (int64_t n = 0; n < rows; ++n)
    for (int64_t k = 0; k < cols; ++k) {
      const uint8_t b = packed[n * (cols / 2) + k / 2];
      q[n * cols + k] = static_cast<int8_t>(int4_value((k % 2 == 0) ? b : (b >> 4)));
    }
}

void oracle_unpack_along_rows(const uint8_t* packed, int64_t rows, int64_t cols, int8_t* q) {
  for (int64_t n = 0; n < rows; ++n)
    for (int64_t k = 0; k < cols; ++k) {
      const uint8_t b = packed[(n / 2) * cols + k];
      q[n * cols + k] = static_cast<int8_t>(int4_value((n % 2 == 0) ? b : (b >> 4)));
    }
}

void oracle_dequant(const uint8_t* packed, const uint16_t* scales, int64_t rows, int64_t cols,
                    int scale_kind, double* out) {
  dequant_matrix(packed, scales, rows, cols, scale_kind, out);
}

void oracle_bf16_encode(const float* in, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_encode(in[i]);
}
void oracle_fp16_encode(const float* in, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = fp16_encode(in[i]);
}
void oracle_fp16_decode(const uint16_t* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = fp16_decode(in[i]);
}

// Route layout.  Valid iff id != -1 and 0 <= id - expert_offset < E.
// counts[e]      routes of local expert e
// offs[e]        start of expert e's segment; segments padded to multiples of bm
// perm[slot]     flat route index t*k + j in the slot, -1 in padding slots
// inv[r]         slot of route r, -1 for invalid/masked routes
// tiles[4*i..]   (expert, first slot, valid rows, 0) for every bm-row tile
// Within an expert, routes keep ascending flat index order (stable).
int oracle_prepare_routes(const int32_t* desc_in, int32_t num_tokens, const int32_t* ids, int32_t bm,
                          int32_t* counts, int32_t* offs, int32_t* perm, int64_t perm_cap,
                          int32_t* inv, int32_t* tiles, int64_t tiles_cap, int32_t* num_tiles) {
  Desc d;
  std::memcpy(&d, desc_in, sizeof(Desc));
  if (bm <= 0 || num_tokens < 0) return 1;
  const int64_t R = static_cast<int64_t>(num_tokens) * d.top_k;
  const int E = d.num_experts;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t r = 0; r < R; ++r) {
    const int l = local_expert(d, ids[r]);
    if (l >= 0) counts[l] += 1;
  }
  offs[0] = 0;
  for (int e = 0; e < E; ++e) {
    const int32_t padded = (counts[e] + bm - 1) / bm * bm;
    offs[e + 1] = offs[e] + padded;
  }
  if (offs[E] > perm_cap) return 2;
  for (int64_t s = 0; s < offs[E]; ++s) perm[s] = -1;
  std::vector<int32_t> next(offs, offs + E);
  for (int64_t r = 0; r < R; ++r) {
    const int l = local_expert(d, ids[r]);
    if (l < 0) {
      inv[r] = -1;
      continue;
    }
    const int32_t slot = next[l]++;
    perm[slot] = static_cast<int32_t>(r);
    inv[r] = slot;
  }
  int64_t nt = 0;
  for (int e = 0; e < E; ++e) {
    for (int32_t m = 0; m < counts[e]; m += bm) {
      if (nt >= tiles_cap) return 3;
      tiles[4 * nt + 0] = e;
      tiles[4 * nt + 1] = offs[e] + m;
      tiles[4 * nt + 2] = (counts[e] - m < bm) ? counts[e] - m : bm;
      tiles[4 * nt + 3] = 0;
      ++nt;
    }
  }
  *num_tiles = static_cast<int32_t>(nt);
  return 0;
}

// Router scores -> routes, the step before the route layout: "feat(pytorch):
// add CuTeDSL W4A16 MoE backend" (LMDeploy), section *Benchmark*, takes the
// routes from a router score / top-k computation (outside its timed region)
// and gives the routing weights as FP32 with renormalize=False.  Plainest
// reading: probabilities p = softmax(logits[t, :]) over all num_global
// experts; the k experts with the largest p, in descending order, ties to the
// lower expert index; weights are those p.  softmax is strictly increasing in
// the logit, so the order is taken on the logits themselves (exact); p is
// computed in double.
int oracle_route_topk(const float* logits, int32_t num_tokens, int32_t num_global, int32_t top_k,
                      int32_t* ids, double* weights) {
  if (num_tokens < 0 || num_global < 1 || top_k < 1 || top_k > num_global) return 1;
  std::vector<int32_t> order(num_global);
  for (int32_t t = 0; t < num_tokens; ++t) {
    const float* l = logits + static_cast<int64_t>(t) * num_global;
    double m = l[0];
    for (int32_t e = 1; e < num_global; ++e) m = l[e] > m ? l[e] : m;
    double sum = 0.0;
    for (int32_t e = 0; e < num_global; ++e) sum += std::exp(static_cast<double>(l[e]) - m);
    // selection: repeatedly take the largest remaining logit (lowest index on ties)
    std::vector<char> taken(num_global, 0);
    for (int32_t j = 0; j < top_k; ++j) {
      int32_t best = -1;
      for (int32_t e = 0; e < num_global; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e;
      }
      taken[best] = 1;
      ids[static_cast<int64_t>(t) * top_k + j] = best;
      weights[static_cast<int64_t>(t) * top_k + j] = std::exp(static_cast<double>(l[best]) - m) / sum;
    }
  }
  return 0;
}

// Masked-count layout ("feat(pytorch): add CuTeDSL W4A16 MoE backend"
// (LMDeploy), section Modification: invalid routes and masked expert counts,
// the layout a low-latency expert-parallel dispatch hands over): the
// activations of local expert e sit in rows [e * max_rows, e * max_rows +
// counts[e]) of an [E * max_rows, H] buffer and the rest is ignored.  As routes:
// row r = e * max_rows + i is one token with a single route, to global expert
// expert_offset + e with weight 1.0, when i < counts[e] (counts clamped to
// [0, max_rows]), else an invalid route (-1).  The forward over these routes
// (top_k = 1) gives every valid row its expert's MLP output and zero rows
// elsewhere.
int oracle_masked_routes(const int32_t* counts, int32_t E, int32_t max_rows, int32_t expert_offset,
                         int32_t* ids, float* weights) {
  if (E < 1 || max_rows < 0) return 1;
  for (int32_t e = 0; e < E; ++e) {
    int32_t c = counts[e];
    if (c < 0) c = 0;
    if (c > max_rows) c = max_rows;
    for (int32_t i = 0; i < max_rows; ++i) {
      const int64_t r = static_cast<int64_t>(e) * max_rows + i;
      ids[r] = i < c ? expert_offset + e : -1;
      weights[r] = 1.0f;
    }
  }
  return 0;
}

// The MoE forward for a subset of tokens (rows == nullptr: all tokens).
// x [T, H] (bf16 or fp16 bits), topk_weights/ids [T, k].
// acc_out [nrows, H] FP32 combine result before the cast; out [nrows, H] bits.
int oracle_moe_forward(const int32_t* desc_in, int32_t num_tokens, const uint16_t* x,
                       const uint8_t* w13, const uint16_t* s13, const uint8_t* w2,
                       const uint16_t* s2, const float* topk_weights, const int32_t* ids,
                       int32_t renormalize, const int32_t* rows, int32_t nrows, float* acc_out,
                       uint16_t* out, int32_t nthreads) {
  Desc d;
  std::memcpy(&d, desc_in, sizeof(Desc));
  const int E = d.num_experts, H = d.hidden, I = d.inter, k = d.top_k;
  const int N1 = d.act == 0 ? 2 * I : I;
  if (rows == nullptr) nrows = num_tokens;
  if (nrows < 0) return 1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
  auto token_of = [&](int64_t i) -> int64_t { return rows ? rows[i] : i; };
  auto act_decode = [&](uint16_t v) { return d.act_dtype == 0 ? bf16_decode(v) : fp16_decode(v); };

  // Routing weights, renormalised over all k entries (FP32, j ascending) when
  // asked; a zero sum gives zero weights.
  std::vector<float> wr(static_cast<size_t>(nrows) * k);
  for (int64_t i = 0; i < nrows; ++i) {
    const int64_t t = token_of(i);
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) sum = sum + topk_weights[t * k + j];
    for (int j = 0; j < k; ++j) {
      const float w = topk_weights[t * k + j];
      wr[i * k + j] = renormalize ? (sum != 0.0f ? w / sum : 0.0f) : w;
    }
  }

  // Routes grouped by local expert, so each expert is dequantised once.
  std::vector<std::vector<int64_t>> by_expert(E);
  for (int64_t i = 0; i < nrows; ++i)
    for (int j = 0; j < k; ++j) {
      const int l = local_expert(d, ids[token_of(i) * k + j]);
      if (l >= 0) by_expert[l].push_back(i * k + j);
    }

  // y[i*k + j][c]: the expert MLP output of each valid route, stored FP32.
  std::vector<float> y(static_cast<size_t>(nrows) * k * H, 0.0f);
  const int64_t w13_sz = d.scale_kind == 0 ? static_cast<int64_t>(N1) * H / 2 : static_cast<int64_t>(N1) / 2 * H;
  const int64_t s13_sz = d.scale_kind == 0 ? static_cast<int64_t>(N1) * (H / 32) : N1;
  const int64_t w2_sz = d.scale_kind == 0 ? static_cast<int64_t>(H) * I / 2 : static_cast<int64_t>(H) / 2 * I;
  const int64_t s2_sz = d.scale_kind == 0 ? static_cast<int64_t>(H) * (I / 32) : H;

#pragma omp parallel
  {
    std::vector<double> W1, W2, xv(H), h(N1), a(I);
#pragma omp for schedule(dynamic, 1)
    for (int e = 0; e < E; ++e) {
      if (by_expert[e].empty()) continue;
      W1.resize(static_cast<size_t>(N1) * H);
      W2.resize(static_cast<size_t>(H) * I);
      dequant_matrix(w13 + e * w13_sz, s13 + e * s13_sz, N1, H, d.scale_kind, W1.data());
      dequant_matrix(w2 + e * w2_sz, s2 + e * s2_sz, H, I, d.scale_kind, W2.data());
      for (int64_t route : by_expert[e]) {
        const int64_t i = route / k;
        const int64_t t = token_of(i);
        for (int c = 0; c < H; ++c) xv[c] = act_decode(x[t * H + c]);
        // gate/up (or fc1) GEMM
        for (int n = 0; n < N1; ++n) {
          double acc = 0.0;
          const double* wrow = &W1[static_cast<size_t>(n) * H];
          for (int c = 0; c < H; ++c) acc += wrow[c] * xv[c];
          h[n] = acc;
        }
        // activation: SwiGLU silu(gate) * up with gate rows first, or relu^2
        for (int n = 0; n < I; ++n) {
          if (d.act == 0) {
            a[n] = silu(h[n]) * h[I + n];
          } else {
            const double r = h[n] > 0.0 ? h[n] : 0.0;
            a[n] = r * r;
          }
        }
        // down GEMM
        for (int c = 0; c < H; ++c) {
          double acc = 0.0;
          const double* wrow = &W2[static_cast<size_t>(c) * I];
          for (int n = 0; n < I; ++n) acc += wrow[n] * a[n];
          y[static_cast<size_t>(route) * H + c] = static_cast<float>(acc);
        }
      }
    }
  }

  // Combine: FP32, fixed top-k order, invalid routes skipped, one cast.
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < nrows; ++i) {
    const int64_t t = token_of(i);
    for (int c = 0; c < H; ++c) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j) {
        if (local_expert(d, ids[t * k + j]) < 0) continue;
        const float prod = wr[i * k + j] * y[(static_cast<size_t>(i) * k + j) * H + c];
        acc = acc + prod;
      }
      if (acc_out) acc_out[i * H + c] = acc;
      if (out) out[i * H + c] = d.act_dtype == 0 ? bf16_encode(acc) : fp16_encode(acc);
    }
  }
  return 0;
}

// Interleaved relayout of packed weights: the layout w4a16_moe_relayout_weights
// documents in include/w4a16_moe.h (the library's own, not the pages'; the
// pages only say the packed INT4 weights are reordered once at setup:
// "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy), Motivation, and
// "[None][feat] Add W4A16 per-channel weight-only support for Cutlass fused
// MoE" (TensorRT-LLM), Changes).  Written out code by code from that
// definition: output rows are packed along K; the code of K index k of row n
// goes to 32-bit word k / 8 of the row, at nibble position p where
// {0, 2, 4, 6, 1, 3, 5, 7}[p] = k % 8 (nibble position p = byte p / 2 of the
// little-endian word, high nibble when p is odd).  Input: the checkpoint
// layout for scale_kind (0: [E, N, K/2] packed along K; 1: [E, N/2, K] packed
// along rows).  Returns 0, or -1 when K is not a multiple of 8 or (row-pair
// input) N is odd.
int oracle_relayout_interleaved(const uint8_t* packed, int32_t scale_kind, int64_t E, int64_t N, int64_t K,
                                uint8_t* out) {
  if (K % 8 != 0 || (scale_kind != 0 && N % 2 != 0)) return -1;
  std::memset(out, 0, static_cast<size_t>(E * N * (K / 2)));
  for (int64_t e = 0; e < E; ++e) {
    for (int64_t n = 0; n < N; ++n) {
      for (int64_t k = 0; k < K; ++k) {
        unsigned code;
        if (scale_kind == 0) {
          const uint8_t b = packed[(e * N + n) * (K / 2) + k / 2];
          code = (k % 2 == 0) ? (b & 0xF) : (b >> 4);
        } else {
          const uint8_t b = packed[(e * (N / 2) + n / 2) * K + k];
          code = (n % 2 == 0) ? (b & 0xF) : (b >> 4);
        }
        const int64_t j = k % 8;
        const int64_t pos = (j % 2 == 0) ? j / 2 : 4 + j / 2;
        uint8_t& dst = out[(e * N + n) * (K / 2) + (k / 8) * 4 + pos / 2];
        dst = static_cast<uint8_t>(dst | ((pos % 2 == 0) ? code : (code << 4)));
      }
    }
  }
  return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
