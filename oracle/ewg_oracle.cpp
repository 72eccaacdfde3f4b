// Plain CPU oracle for sparse embedding weight-gradient accumulation.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
// this file: only the tests, the smoke check and the bench's CPU-baseline arm.
// It shares no code, header, table or helper with the CUDA library.
//
// What it computes (Megatron Core API docs, core.fusions.fused_embedding_wgrad,
// module docstring and the accumulate_embedding_wgrad entry):
//
//   main_grad += embedding_dense_backward(grad, ids), touching only rows of ids.
//
// in exactly the order the module docstring gives for PyTorch's sort-based
// embedding backward followed by main_grad.add_:
//
//   1. sort the token ids together with their positions            (docstring, 1st bullet)
//   2. per token, sum its gradient rows in position order into fp32 partial
//      sums of at most NROWS = 10 rows; chunks start at the token's first row
//   3. add those partial sums in order, starting from +0.0f
//   4. round once to the gradient dtype
//   5. add that to the main_grad row in fp32, round to main_grad's dtype  (2nd bullet)
//   6. rows of tokens that do not occur are neither read nor written    (docstring, last line)
//
// Floating point: IEEE binary32 adds in round-to-nearest-even, no FMA (there are
// no products), no flush-to-zero.  Build with -O2 -ffp-contract=off and never with
// -ffast-math.  fp32 -> bf16 rounding is written out from the IEEE-754 encoding.
//
// Parity: pinned (see the "not gpu" oracle tests: closed forms, integer sums,
// an fp64 error bound, hand-derived order cases, library rounding).

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <thread>
#include <utility>
#include <vector>

namespace {

constexpr int kNrows = 10;  // partial-sum chunk length (NROWS_PER_THREAD on the page)

enum DType { kInt32 = 0, kInt64 = 1, kBf16 = 2, kFp32 = 3 };
enum Result { kOk = 0, kInvalid = 2, kIdOutOfRange = 4 };

// --- element conversions ---------------------------------------------------

float bf16_to_float(uint16_t b) {
  // a bf16 value is the upper half of the binary32 encoding
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

uint16_t float_to_bf16(float f) {
  // Round-to-nearest, ties-to-even, on the 16 low bits of the binary32 encoding.
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  const bool is_nan = (u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0;
  if (is_nan) {
    // keep sign and upper payload, force the quiet bit so the result stays NaN
    return static_cast<uint16_t>((u >> 16) | 0x0040u);
  }
  uint32_t kept = u >> 16;          // sign, exponent, 7 fraction bits
  uint32_t dropped = u & 0xffffu;   // the 16 bits that are rounded away
  const uint32_t half = 0x8000u;
  if (dropped > half || (dropped == half && (kept & 1u))) {
    kept += 1;  // a carry out of the fraction bumps the exponent (up to +inf)
  }
  return static_cast<uint16_t>(kept);
}

float load_elem(const void* base, int dtype, int64_t index) {
  if (dtype == kBf16) return bf16_to_float(static_cast<const uint16_t*>(base)[index]);
  return static_cast<const float*>(base)[index];
}

// The single rounding of a token's summed row to the gradient's dtype (Megatron Core API
// docs, core.fusions.fused_embedding_wgrad, module docstring, first bullet); returns the
// rounded value widened back to float.
float round_to(int dtype, float x) {
  if (dtype == kBf16) return bf16_to_float(float_to_bf16(x));
  return x;  // fp32 -> fp32 is the identity
}

void store_elem(void* base, int dtype, int64_t index, float x) {
  if (dtype == kBf16) {
    static_cast<uint16_t*>(base)[index] = float_to_bf16(x);
  } else {
    static_cast<float*>(base)[index] = x;
  }
}

int64_t load_id(const void* ids, int dtype, int64_t p) {
  if (dtype == kInt32) return static_cast<const int32_t*>(ids)[p];
  return static_cast<const int64_t*>(ids)[p];
}

// --- step 1: sort (token, position) pairs -----------------------------------

struct Run {
  int64_t id;
  int64_t first;  // index into the sorted pair list
  int64_t length;
};

// Returns the sorted positions (grouped by id, positions ascending within an id)
// and the list of runs.  A library sort serves as the step: pairs (id, position)
// are unique, so sorting them lexicographically is the stable sort by id.
void sort_pairs(const std::vector<int64_t>& id_of, std::vector<int64_t>& sorted_pos,
                std::vector<Run>& runs) {
  const int64_t n = static_cast<int64_t>(id_of.size());
  std::vector<std::pair<int64_t, int64_t>> pairs(n);
  for (int64_t p = 0; p < n; ++p) pairs[p] = {id_of[p], p};
  std::sort(pairs.begin(), pairs.end());
  sorted_pos.resize(n);
  runs.clear();
  for (int64_t s = 0; s < n; ++s) {
    sorted_pos[s] = pairs[s].second;
    if (s == 0 || pairs[s].first != pairs[s - 1].first) {
      runs.push_back({pairs[s].first, s, 0});
    }
    runs.back().length += 1;
  }
}

// --- steps 2-4: one token's weight-gradient row -----------------------------

struct GradView {
  const void* data;
  int dtype;
  int64_t row_stride;  // elements between consecutive token rows
};

// Writes w[h] = round_g( ((0 + P_0) + P_1) + ... ), P_c = ((0 + g_{10c}) + g_{10c+1}) + ...
// where g_k is the gradient row of the k-th occurrence of the token (position order).
void run_weight_grad(const Run& run, const std::vector<int64_t>& sorted_pos,
                     const GradView& g, int64_t H, std::vector<float>& total,
                     std::vector<float>& part, float* w_out) {
  // the partial sums are combined in chunk order, beginning from zero (module docstring,
  // first bullet)
  total.assign(H, 0.0f);
  for (int64_t c0 = 0; c0 < run.length; c0 += kNrows) {
    const int64_t c1 = std::min<int64_t>(c0 + kNrows, run.length);
    part.assign(H, 0.0f);  // each partial sum starts at +0
    for (int64_t k = c0; k < c1; ++k) {
      const int64_t pos = sorted_pos[run.first + k];
      const int64_t row = pos * g.row_stride;
      for (int64_t h = 0; h < H; ++h) {
        part[h] = part[h] + load_elem(g.data, g.dtype, row + h);
      }
    }
    for (int64_t h = 0; h < H; ++h) total[h] = total[h] + part[h];
  }
  for (int64_t h = 0; h < H; ++h) w_out[h] = round_to(g.dtype, total[h]);
}

// Splits runs into contiguous groups of roughly equal row counts, one per thread.
// Runs are independent, so the split does not change any value.
template <typename Fn>
void for_runs_parallel(const std::vector<Run>& runs, int64_t n, int num_threads, Fn fn) {
  unsigned hw = std::thread::hardware_concurrency();
  int t = num_threads > 0 ? num_threads : static_cast<int>(hw == 0 ? 1 : hw);
  if (t > static_cast<int>(runs.size())) t = static_cast<int>(runs.size());
  if (t <= 1) {
    fn(static_cast<size_t>(0), runs.size());
    return;
  }
  std::vector<size_t> bounds(t + 1, runs.size());
  bounds[0] = 0;
  int64_t seen = 0;
  int next = 1;
  for (size_t r = 0; r < runs.size() && next < t; ++r) {
    seen += runs[r].length;
    if (seen * t >= n * next) bounds[next++] = r + 1;
  }
  std::vector<std::thread> pool;
  for (int i = 0; i < t; ++i) pool.emplace_back(fn, bounds[i], bounds[i + 1]);
  for (auto& th : pool) th.join();
}

int read_ids(const void* ids, int ids_dtype, int64_t n, int64_t V, std::vector<int64_t>& out) {
  if (ids_dtype != kInt32 && ids_dtype != kInt64) return kInvalid;
  out.resize(n);
  for (int64_t p = 0; p < n; ++p) {
    const int64_t id = load_id(ids, ids_dtype, p);
    if (id < 0 || id >= V) return kIdOutOfRange;
    out[p] = id;
  }
  return kOk;
}

bool float_dtype(int d) { return d == kBf16 || d == kFp32; }

}  // namespace

extern "C" {

// main_grad[V][H] (row stride mg_row_stride) += embedding_dense_backward(grad, ids),
// touching only rows whose id occurs.  grad is [n][H] with row stride grad_row_stride.
// Returns 0, 2 (bad arguments) or 4 (an id outside [0, V)); main_grad is unchanged
// on error.  num_threads <= 0 uses every hardware thread.
int ewg_oracle_accumulate(const void* ids, int ids_dtype, int64_t n, const void* grad,
                          int grad_dtype, int64_t grad_row_stride, void* main_grad,
                          int mg_dtype, int64_t V, int64_t H, int64_t mg_row_stride,
                          int num_threads) {
  if (n < 0 || V < 1 || H < 1 || !float_dtype(grad_dtype) || !float_dtype(mg_dtype) ||
      grad_row_stride < H || mg_row_stride < H)
    return kInvalid;
  std::vector<int64_t> id_of;
  int rc = read_ids(ids, ids_dtype, n, V, id_of);
  if (rc != kOk) return rc;
  std::vector<int64_t> sorted_pos;
  std::vector<Run> runs;
  sort_pairs(id_of, sorted_pos, runs);
  const GradView g{grad, grad_dtype, grad_row_stride};
  for_runs_parallel(runs, n, num_threads, [&](size_t r0, size_t r1) {
    std::vector<float> total, part, w(H);
    for (size_t r = r0; r < r1; ++r) {
      run_weight_grad(runs[r], sorted_pos, g, H, total, part, w.data());
      // main_grad.add_(w): fp32 add, round to main_grad's dtype
      const int64_t row = runs[r].id * mg_row_stride;
      for (int64_t h = 0; h < H; ++h) {
        const float m = load_elem(main_grad, mg_dtype, row + h);
        store_elem(main_grad, mg_dtype, row + h, m + w[h]);
      }
    }
  });
  return kOk;
}

// The weight-gradient rows themselves (steps 1-4, before the add into main_grad):
// writes the U distinct ids in ascending order to uniq_ids[0..U) and their rows,
// already rounded to the gradient dtype and widened to float, to w[U][H].
// Both outputs need room for n entries.  Returns U, or -2 / -4 on error.
int64_t ewg_oracle_weight_grad(const void* ids, int ids_dtype, int64_t n, const void* grad,
                               int grad_dtype, int64_t grad_row_stride, int64_t V, int64_t H,
                               int64_t* uniq_ids, float* w, int num_threads) {
  if (n < 0 || V < 1 || H < 1 || !float_dtype(grad_dtype) || grad_row_stride < H)
    return -kInvalid;
  std::vector<int64_t> id_of;
  int rc = read_ids(ids, ids_dtype, n, V, id_of);
  if (rc != kOk) return -rc;
  std::vector<int64_t> sorted_pos;
  std::vector<Run> runs;
  sort_pairs(id_of, sorted_pos, runs);
  const GradView g{grad, grad_dtype, grad_row_stride};
  for_runs_parallel(runs, n, num_threads, [&](size_t r0, size_t r1) {
    std::vector<float> total, part;
    for (size_t r = r0; r < r1; ++r) {
      uniq_ids[r] = runs[r].id;
      run_weight_grad(runs[r], sorted_pos, g, H, total, part, w + r * H);
    }
  });
  return static_cast<int64_t>(runs.size());
}

// Sorted (id, position) pairs as the oracle forms them (step 1 alone).
int ewg_oracle_sort_pairs(const void* ids, int ids_dtype, int64_t n, int64_t V,
                          int64_t* sorted_ids, int64_t* sorted_pos) {
  std::vector<int64_t> id_of;
  int rc = read_ids(ids, ids_dtype, n, V, id_of);
  if (rc != kOk) return rc;
  std::vector<int64_t> pos;
  std::vector<Run> runs;
  sort_pairs(id_of, pos, runs);
  for (int64_t s = 0; s < n; ++s) {
    sorted_pos[s] = pos[s];
    sorted_ids[s] = id_of[pos[s]];
  }
  return kOk;
}

// fp32 -> bf16 bits, round-to-nearest-even (the conversion used for both roundings).
void ewg_oracle_round_to_bf16(const float* x, uint16_t* out, int64_t count) {
  for (int64_t i = 0; i < count; ++i) out[i] = float_to_bf16(x[i]);
}

}  // extern "C"
