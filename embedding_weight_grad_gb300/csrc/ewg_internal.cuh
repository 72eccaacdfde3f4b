// Internal declarations shared by the library's translation units.
//
// Vocabulary.  A "run" is the set of sorted slots of one token id; its slots hold the
// token's positions in ascending order.  A "chunk" is up to NROWS consecutive slots of
// a run, counted from the run's first slot.  A run is "long" when it has more than
// NROWS slots (more than one chunk).
//
// Work lists the plan leaves in the caller's workspace, grouped in partitions (one
// partition on the multi-tile path, one per hash partition of the ids otherwise):
//   long chunks   descriptors of every chunk of every long run
//   short chunks  descriptors of the single chunk of every other run
//   long runs     (first partial row, number of chunks C, id) per long run
// A partition's lists are contiguous; per-partition counts and offsets sit in the
// partition tables.  The apply kernels walk the lists partition by partition.
//
// Workspace layout (each region 256-byte aligned):
//   Header | tables | keys/vals x2 (multi-tile sort) | chunk descriptors | run table |
//   tile scratch (histograms, bad-id counts, listing counts) | fp32 partial rows
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace ewg {

constexpr int kNrows = 10;           // chunk length: NROWS_PER_THREAD of PyTorch's backward

// Chunk descriptor: 16 x int32 = 64 bytes.
constexpr int kChunkWords = 16;
constexpr int kDescPos = 0;          // words 0..9: token positions, in position order
constexpr int kDescId = 10;          // token id (main_grad row)
constexpr int kDescMeta = 11;        // len | (c << 4), c = chunk index within the run
constexpr int kDescPartial = 12;     // partial row of this chunk (long runs), else -1
constexpr int kDescNumChunks = 13;   // C, chunks of the run

// Long-run table entry: 4 x int32: first partial row, C, id, q | (split << 4).  A run of
// many chunks is listed `split` times (q = 0..split-1); entry q folds the q-th of
// `split` equal column slices of every 512-column group, so the long folds of heavy runs
// spread over several CTAs.
constexpr int kRunWords = 4;

__host__ __device__ inline int fold_entries(int chunks) {
  return chunks > 64 ? 4 : chunks > 32 ? 2 : 1;
}

// Partition tables: kTables arrays of kMaxParts ints.
constexpr int kMaxParts = 128;
enum Table { kLongCnt = 0, kLongOff, kShortCnt, kShortOff, kRunCnt, kRunOff, kTables };

// Hashed plan (up to 8192 tokens): one CTA per hash partition of the ids.
constexpr int kHashParts = 64;
constexpr int kHashThreads = 1024;
constexpr int kHashItems = 8;
constexpr int kHashMaxN = kHashThreads * kHashItems;      // 8192 tokens
constexpr int kMaxDigitBits = 9;                          // 512 buckets per radix pass

// Multi-tile plan: tiles of kTile keys, one CTA each (each kernel picks its own threads
// per tile).
constexpr int kTile = 2048;
constexpr int kMaxPasses = 4;                             // ids below 2^31: 31 bits, 9 per pass
// Look-back words of the listing: each tile's three words sit in a 128-byte line of their
// own, so the many threads that poll their predecessors spread over L2 slices instead of
// all polling the same few lines.
constexpr int kStatusWords = 32;

// Apply kernel.  Bulk copies reach full HBM bandwidth only from about 4 KB up, so an
// item covers a chunk over a column tile of up to 2048 columns (1024 for an fp32
// gradient), each grad row segment and the main_grad segment one copy.
constexpr int kMaxTileColsBf16 = 2048;
constexpr int kMaxTileColsFp32 = 1024;
constexpr int kCombineCols = 512;     // columns of one combine task (2 KB partial rows)
constexpr int kCombineBatch = 8;      // partial rows per combine ring item
constexpr int kApplyCtasPerSm = 4;    // independent copy-issuing streams per SM
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;           // 8 columns each per pass
constexpr int kApplyThreads = kConsumers + 32;            // + one producer warp
constexpr int kRingBytes = 50 * 1024;
constexpr int kSlots = 16;

// While the plan runs, HBM is nearly idle and the apply CTAs that launched early on the
// SMs it leaves free have nothing to do: they pull up to this many bytes of grad rows
// into L2 (every grad row is read once later, in an order only the plan knows), with a
// keep hint so the rows survive until they are copied.  Measured on GB300: 40 MiB saves
// about 4 us of 68 per call at 8192 x 7168 and 18 us of 1344 at 131072 x 8192; more
// than about 60 MiB crowds L2 and costs time.
constexpr long long kPrefetchBytes = 40ll << 20;

// Column limit of a long-run chunk item (it carries 10 rows).
constexpr int kMaxLongTileCols = 2048;

// Column tile of the chunk items: the widest tile within the limit, split evenly.
inline int tile_cols(int64_t hidden, bool grad_bf16, bool long_chunks) {
  int64_t lim = grad_bf16 ? kMaxTileColsBf16 : kMaxTileColsFp32;
  if (long_chunks && lim > kMaxLongTileCols) lim = kMaxLongTileCols;
  const int64_t tiles = (hidden + lim - 1) / lim;
  const int64_t per = (hidden + tiles - 1) / tiles;
  return static_cast<int>((per + 7) / 8 * 8);
}

enum DeviceStatus { kStatusOk = 0, kStatusInvalid = 2, kStatusBadId = 4, kStatusTimeout = 5, kStatusBounds = 6 };

struct Header {
  int status;            // EWG_OK or the device-detected error of the last call
  int n;                 // stamp of the plan: tokens, hidden, num_embeddings
  int hidden;
  int num_parts;
  long long num_embeddings;
  int bad_ids;
  int work[2];           // next work item of the apply kernel (zeroed by the plan)
  int done;              // apply CTAs that have finished (zeroed by the plan)
  int epoch;             // apply calls completed on this plan (zeroed by the plan)
  int spin_limit;        // polls of a fold's arrival counter before it gives up (set by
                         // the plan to kFoldSpinLimit)
  int pad[52];
};
static_assert(sizeof(Header) == 256, "header is one 256-byte region");
// The GPU tests of the timeout path overwrite these two fields between ewg_plan and
// ewg_apply (an unreachable epoch and a short limit), so their offsets are fixed.
static_assert(offsetof(Header, epoch) == 40 && offsetof(Header, spin_limit) == 44,
              "header offsets the timeout tests rely on");

// Default bound on the polls of a fold's arrival counter (each poll is an L2 round trip
// plus a short sleep: a few seconds in all, far beyond any legitimate wait).
constexpr int kFoldSpinLimit = 1 << 22;

// Index checks of the bounds-checking build (compiled with EWG_DEBUG): returns `ok`, and
// a false one records EWG_ERR_BOUNDS in the status word, after which the caller replaces
// the access by a safe one (row or slot 0).  In the ordinary build every index is
// trusted and the check compiles to nothing.
#ifdef EWG_DEBUG
__device__ __forceinline__ bool checked(bool ok, const Header* h) {
  if (!ok) atomicExch(const_cast<int*>(&h->status), kStatusBounds);
  return ok;
}
#else
__device__ __forceinline__ bool checked(bool, const Header*) { return true; }
#endif

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// fp32 partial rows, kept slice-major per run: the run whose first partial row is p0
// owns floats [p0 P, (p0 + C) P) of the region, P = partial_row_floats(hidden); in
// them, column slice [s, s + w) (w = kCombineCols / fold_entries(C), s a multiple of w)
// of chunk c sits at C s + c w.  A fold batch (consecutive chunks, one slice) is then
// one contiguous block.
__host__ __device__ inline int64_t partial_row_floats(int64_t hidden) {
  return (hidden + kCombineCols - 1) / kCombineCols * kCombineCols;
}

// Long runs of L >= 11 rows have ceil(L/10) <= 2L/11 chunks; partition b of the hashed
// plan starts its partial rows at floor(2 S_b / 11) + b (S_b: tokens of partitions < b).
inline int64_t max_partial_rows(int64_t n) { return 2 * n / 11 + kMaxParts + 1; }
// Table entries: a run of L >= 11 rows has at most L/11 + L/100 of them (one per run, two
// above 320 rows, four above 640); partition b of the hashed plan starts its entries at
// floor(S_b / 11) + floor(S_b / 100) + b.
inline int64_t max_long_runs(int64_t n) { return n / 11 + n / 100 + kMaxParts + 1; }

struct Layout {
  size_t header, tables, keys_a, vals_a, keys_b, vals_b, chunks, runs, tile_hist, ctl, tile_bad, list_status,
      arrivals, partial, total;
  int64_t n, hidden, tiles;
  int64_t short_base;   // multi-tile plan: descriptor index of the first short chunk
};

inline Layout make_layout(int64_t n, int64_t hidden) {
  Layout L{};
  L.n = n;
  L.hidden = hidden;
  L.tiles = ceil_div(n, kTile);
  const int64_t n_pad = L.tiles * kTile;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.header = take(sizeof(Header));
  L.tables = take(sizeof(int) * kTables * kMaxParts);
  L.keys_a = take(n_pad * 4);
  L.vals_a = take(n_pad * 4);
  L.keys_b = take(n_pad * 4);
  L.vals_b = take(n_pad * 4);
  // Chunk descriptors.  The hashed plan uses the first n; the multi-tile plan puts the long
  // runs' chunks first (at most max_partial_rows(n) of them) and the short chunks after.
  L.short_base = max_partial_rows(n);
  L.chunks = take(static_cast<size_t>(L.short_base + n) * kChunkWords * 4);
  L.runs = take(static_cast<size_t>(max_long_runs(n)) * kRunWords * 4);
  L.tile_hist = take(static_cast<size_t>(kMaxPasses) * L.tiles * (1 << kMaxDigitBits) * 4);
  L.ctl = take(static_cast<size_t>(kMaxPasses + 1) * 4);
  L.tile_bad = take(static_cast<size_t>(L.tiles) * 4);
  L.list_status = take(static_cast<size_t>(L.tiles) * kStatusWords * 4);
  L.arrivals = take(static_cast<size_t>(max_partial_rows(n)) * 4);
  L.partial = take(static_cast<size_t>(max_partial_rows(n)) * partial_row_floats(hidden) * 4);
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

// Sort plan for keys in [0, max_key].
inline SortPlan make_sort_plan(int64_t max_key) {
  SortPlan s{};
  s.id_bits = bit_width(static_cast<uint64_t>(max_key));
  s.passes = static_cast<int>(ceil_div(s.id_bits, kMaxDigitBits));
  s.digit_bits = s.passes ? static_cast<int>(ceil_div(s.id_bits, s.passes)) : 0;
  return s;
}

struct PlanArgs {
  const void* ids;
  int ids_int64;
  int n;
  long long num_embeddings;   // ids outside [0, num_embeddings) are errors
  long long row_begin;        // the rows kept: [row_begin, row_begin + shard_rows); an id
  long long shard_rows;       // there becomes key id - row_begin, other ids are skipped
  uint32_t skip_key;          // sort key of a skipped id (shard_rows when sharded)
  int hidden;
  int id_bits, passes, digit_bits;
  int tiles;
  Header* header;
  int* tables;           // [kTables][kMaxParts]
  uint32_t* keys_a;
  uint32_t* vals_a;
  uint32_t* keys_b;
  uint32_t* vals_b;
  int* chunks;
  int chunk_cap;         // descriptors, long-run table entries and partial rows the
  int run_cap;           // workspace holds (checked by the bounds-checking build)
  int partial_cap;
  int short_base;        // multi-tile plan: descriptor index of the first short chunk
  int* runs;
  uint32_t* tile_hist;   // [pass][tile][digit]: keys of each digit in each tile of the pass
  uint32_t* counters;    // [kMaxPasses]: tiles claimed by the listing
  int* tile_bad;         // per tile: ids outside [0, num_embeddings)
  uint32_t* list_status; // per tile, kStatusWords words: look-back words of long chunks, short
                         // chunks, long runs (the first three)
  int* arrivals;         // per long run, at its first partial row: zeroed here
};

struct ApplyArgs {
  const void* grad;
  long long grad_stride;   // elements
  void* main_grad;
  long long mg_stride;     // elements
  int n;
  int hidden;
  int tile_cols_long;      // columns of a long-run chunk item (multiple of 8)
  int tile_cols_rest;      // columns of a short-run chunk item (multiple of 8)
  long long num_embeddings;
  const Header* header;
  const int* tables;
  const int* chunks;
  const int* runs;
  float* partial;
  int partial_cap;         // partial rows the workspace holds
  int* arrivals;           // per long run (at its first partial row): finished chunk parts
  int prefetch_rows;       // grad rows [0, prefetch_rows) pulled into L2 before the kernel
                           // waits on the plan (0: none)
  int parts;               // partitions the plan of n tokens writes (kHashParts or 1)
};

// Detail of the last error on the calling thread (read back by ewg_last_error).
void set_last_error(const char* msg);

// Host-side launchers.
cudaError_t prepare_kernels();   // once per device, before the first launch
cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream);
#ifdef EWG_DEBUG
// The look-back test probe of the bounds-checking build (see include/ewg_debug.h).
cudaError_t launch_lookback_probe(uint32_t* words, int tile, int poll_limit, int* out, cudaStream_t stream);
#endif
// The apply kernel, chained to its predecessor by programmatic dependent launch.
cudaError_t launch_apply(const ApplyArgs& a, int grad_bf16, int mg_bf16, int num_sms,
                         cudaStream_t stream);

}  // namespace ewg
