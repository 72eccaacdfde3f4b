// Internal declarations shared by the library's translation units.
//
// Data layout in the caller's workspace (each region 256-byte aligned):
//
//   Header        status words, chunk counts and the stamp of the plan
//   keys/vals x2  ping-pong buffers of the radix sort: id (u32) and position (u32)
//   chunks        one 64-byte descriptor per chunk: up to 10 token positions, the id,
//                 chunk index c within its run, chunks in the run C, and the index
//                 of its fp32 partial row when the run is long
//   tile scratch  per-tile digit histograms, bad-id counts and listing counts
//   counters      one arrival counter per (long-run chunk, 256-column slice)
//   partial       fp32 [max long-run chunks][hidden] chunk partial sums
//
// A "chunk" is up to NROWS consecutive sorted slots of one token's run, counted from
// the run's first slot; a run is "long" when it has more than NROWS slots.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace ewg {

constexpr int kNrows = 10;           // chunk length: NROWS_PER_THREAD of PyTorch's backward
constexpr int kSliceCols = 256;      // columns one warp covers (32 lanes x 8 elements)
constexpr int kChunkWords = 16;      // 64-byte chunk descriptor
constexpr int kDescPos = 0;          // words 0..9: token positions, in position order
constexpr int kDescId = 10;          // word 10: the token id (main_grad row)
constexpr int kDescMeta = 11;        // word 11: len | (c << 4)
constexpr int kDescLong = 12;        // word 12: partial row of this chunk, -1 for short runs
constexpr int kDescNumChunks = 13;   // word 13: C, the number of chunks of the run

// Single-CTA plan (sort + listing entirely in shared memory).
constexpr int kSmallThreads = 1024;
constexpr int kSmallItems = 8;
constexpr int kSmallMaxN = kSmallThreads * kSmallItems;   // 8192 tokens
constexpr int kMaxDigitBits = 9;                          // 512 buckets per radix pass

// Multi-CTA plan.
constexpr int kTileThreads = 256;
constexpr int kTileItems = 8;
constexpr int kTile = kTileThreads * kTileItems;          // 2048 keys per tile

// Apply kernel.
constexpr int kApplyThreads = 256;

struct Header {
  int status;            // EWG_OK or the device-detected error of the last call
  int num_chunks;
  int num_long_chunks;
  int bad_ids;
  int n;                 // stamp of the plan: tokens, hidden, num_embeddings
  int hidden;
  long long num_embeddings;
  int pad[56];
};
static_assert(sizeof(Header) == 256, "header is one 256-byte region");

struct Layout {
  size_t header, keys_a, vals_a, keys_b, vals_b, chunks, hist, tile_bad, tile_cnt, counters,
      partial, total;
  int64_t n, hidden, tiles, slices, max_long_chunks;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Every long run of L >= 11 rows has ceil(L/10) <= 2L/11 chunks.
inline int64_t max_long_chunks(int64_t n) { return 2 * n / 11 + 1; }

inline Layout make_layout(int64_t n, int64_t hidden) {
  Layout L{};
  L.n = n;
  L.hidden = hidden;
  L.tiles = ceil_div(n, kTile);
  L.slices = ceil_div(hidden, kSliceCols);
  L.max_long_chunks = max_long_chunks(n);
  const int64_t n_pad = L.tiles * kTile;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.header = take(sizeof(Header));
  L.keys_a = take(n_pad * 4);
  L.vals_a = take(n_pad * 4);
  L.keys_b = take(n_pad * 4);
  L.vals_b = take(n_pad * 4);
  L.chunks = take(static_cast<size_t>(n) * kChunkWords * 4);
  L.hist = take(static_cast<size_t>(L.tiles) * (1 << kMaxDigitBits) * 4);
  L.tile_bad = take(static_cast<size_t>(L.tiles) * 4);
  L.tile_cnt = take(static_cast<size_t>(L.tiles) * 8);
  L.counters = take(static_cast<size_t>(L.max_long_chunks) * L.slices * 4);
  L.partial = take(static_cast<size_t>(L.max_long_chunks) * hidden * 4);
  L.total = off;
  return L;
}

// Radix passes over the id bits only: the input is already in position order and an
// LSD radix sort is stable, so positions need no passes of their own.
struct SortPlan {
  int id_bits;
  int passes;
  int digit_bits;
};

inline int bit_width(uint64_t x) {
  int b = 0;
  while (x) {
    ++b;
    x >>= 1;
  }
  return b;
}

inline SortPlan make_sort_plan(int64_t num_embeddings) {
  SortPlan s{};
  s.id_bits = bit_width(static_cast<uint64_t>(num_embeddings - 1));
  s.passes = static_cast<int>(ceil_div(s.id_bits, kMaxDigitBits));
  s.digit_bits = s.passes ? static_cast<int>(ceil_div(s.id_bits, s.passes)) : 0;
  return s;
}

// Arguments of the plan kernels.
struct PlanArgs {
  const void* ids;
  int ids_int64;
  int n;
  long long num_embeddings;
  int hidden;
  int slices;
  int id_bits, passes, digit_bits;
  int tiles;
  Header* header;
  uint32_t* keys_a;
  uint32_t* vals_a;
  uint32_t* keys_b;
  uint32_t* vals_b;
  int* chunks;
  uint32_t* hist;
  int* tile_bad;
  long long* tile_cnt;
  int* counters;
};

// Arguments of the apply kernel.
struct ApplyArgs {
  const void* grad;
  long long grad_stride;   // elements
  void* main_grad;
  long long mg_stride;     // elements
  int n;
  int hidden;
  long long num_embeddings;
  int slices;
  const Header* header;
  const int* chunks;
  int* counters;
  float* partial;
};

// Host-side launchers (each returns cudaSuccess or the launch error).
cudaError_t prepare_plan_kernels();   // once per device, before the first launch
cudaError_t launch_plan(const PlanArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_apply(const ApplyArgs& a, int grad_bf16, int mg_bf16, int num_sms,
                         cudaStream_t stream);

}  // namespace ewg
