// Plan kernels: id validation, (token, position) sort and run / chunk listing.
//
// Counterpart of _sort_tokens_kernel (Megatron Core API docs,
// core.fusions.fused_embedding_wgrad, "Functions"): sort the (token, position) pairs,
// find every sorted slot's run, list the chunks of at most NROWS slots.
//
// The sort is an LSD radix sort over the id bits only.  Keys arrive in position
// order and every pass is stable, so positions stay ascending inside each run
// without passes of their own.  Up to 8192 tokens one CTA does everything in
// shared memory; above that the passes run as histogram / scan / scatter kernels
// over tiles of 2048 keys.
//
// The listing gives every sorted slot s its run's first slot rs and last slot re.
// Slot s starts a chunk when (s - rs) % NROWS == 0; chunks are numbered by a scan
// in slot order, and chunks of runs longer than NROWS also get a row of the fp32
// partial-sum buffer.  Each chunk is written as a 64-byte descriptor that carries
// its token positions, so the apply kernel needs no further indirection.
#include <climits>

#include "ewg.h"
#include "ewg_internal.cuh"

namespace ewg {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kPadKey = 0xffffffffu;  // sorts after every id in every pass

struct MaxOp {
  __device__ int operator()(int a, int b) const { return a > b ? a : b; }
};
struct MinOp {
  __device__ int operator()(int a, int b) const { return a < b ? a : b; }
};
struct SumOp {
  __device__ long long operator()(long long a, long long b) const { return a + b; }
};

// Exclusive prefix scan over the block in thread order.  `sw` needs NW entries.
template <int NT, typename T, typename Op>
__device__ T block_exclusive_scan(T v, Op op, T ident, T* sw, T* total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x = op(y, x);
  }
  if (lane == 31) sw[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T a = lane < NW ? sw[lane] : ident;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_up_sync(kFull, a, o);
      if (lane >= o) a = op(y, a);
    }
    if (lane < NW) sw[lane] = a;
  }
  __syncthreads();
  T before_warp = warp > 0 ? sw[warp - 1] : ident;
  T up = __shfl_up_sync(kFull, x, 1);
  T excl = op(before_warp, lane > 0 ? up : ident);
  if (total) *total = sw[NW - 1];
  __syncthreads();
  return excl;
}

// Exclusive suffix scan: combines the values of all threads after this one.
template <int NT, typename T, typename Op>
__device__ T block_exclusive_suffix_scan(T v, Op op, T ident, T* sw) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_down_sync(kFull, x, o);
    if (lane + o < 32) x = op(x, y);
  }
  if (lane == 0) sw[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T a = lane < NW ? sw[lane] : ident;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_down_sync(kFull, a, o);
      if (lane + o < 32) a = op(a, y);
    }
    if (lane < NW) sw[lane] = a;
  }
  __syncthreads();
  T after_warp = warp + 1 < NW ? sw[warp + 1] : ident;
  T down = __shfl_down_sync(kFull, x, 1);
  T excl = op(lane < 31 ? down : ident, after_warp);
  __syncthreads();
  return excl;
}

template <int NT>
__device__ int block_sum_int(int v, long long* sw64) {
  long long tot = 0;
  block_exclusive_scan<NT, long long>(static_cast<long long>(v), SumOp(), 0ll, sw64, &tot);
  return static_cast<int>(tot);
}

__device__ __forceinline__ long long load_id(const void* ids, int is64, int i) {
  return is64 ? static_cast<const long long*>(ids)[i] : static_cast<const int*>(ids)[i];
}

// Validated sort key of token i: the id, 0 for an out-of-range id (the call is then
// void anyway), kPadKey past the end.
__device__ __forceinline__ uint32_t make_key(const PlanArgs& a, int i, int& bad) {
  if (i >= a.n) return kPadKey;
  long long id = load_id(a.ids, a.ids_int64, i);
  if (id < 0 || id >= a.num_embeddings) {
    ++bad;
    return 0u;
  }
  return static_cast<uint32_t>(id);
}

// Warp-wide 32-ary search in a sorted key array: first index in [lo, hi) whose key
// is >= k (upper == false) or > k (upper == true); hi if there is none.
__device__ int warp_bound(const uint32_t* keys, int lo, int hi, uint32_t k, bool upper) {
  const int lane = threadIdx.x & 31;
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    bool pred = true;  // probes past hi count as "beyond"
    if (idx < hi) {
      const uint32_t v = keys[idx];
      pred = upper ? (v > k) : (v >= k);
    }
    const unsigned m = __ballot_sync(kFull, pred);
    const int f = m ? __ffs(m) - 1 : 32;
    const int nlo = f > 0 ? lo + (f - 1) * step + 1 : lo;
    const int nhi = f < 32 ? min(hi, lo + f * step) : hi;
    lo = nlo;
    hi = nhi;
  }
  const int idx = lo + lane;
  bool pred = true;
  if (idx < hi) {
    const uint32_t v = keys[idx];
    pred = upper ? (v > k) : (v >= k);
  }
  const unsigned m = __ballot_sync(kFull, pred);
  const int f = m ? __ffs(m) - 1 : 32;
  return min(lo + f, hi);
}

// ---------------------------------------------------------------------------
// Listing of one block of slots [s_begin, s_begin + NT*ITEMS), thread-blocked.
// rs_seed: first slot of the run of slot s_begin; re_seed: last slot of the run of
// the block's last valid slot.  Produces per-item run bounds in registers.
template <int NT, int ITEMS>
struct Listing {
  int rs[ITEMS];
  int re[ITEMS];
  uint32_t key[ITEMS];

  __device__ void compute(const uint32_t* keys, int n, int s_begin, int rs_seed, int re_seed,
                          int* swi) {
    const int base = s_begin + threadIdx.x * ITEMS;
    bool head[ITEMS], tail[ITEMS];
    int hmax = -1, tmin = INT_MAX;
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int s = base + i;
      head[i] = tail[i] = false;
      key[i] = kPadKey;
      if (s < n) {
        key[i] = keys[s];
        head[i] = (s == 0) || keys[s - 1] != key[i];
        tail[i] = (s == n - 1) || keys[s + 1] != key[i];
        if (head[i]) hmax = max(hmax, s);
        if (tail[i]) tmin = min(tmin, s);
      }
    }
    int before = block_exclusive_scan<NT, int>(hmax, MaxOp(), -1, swi, nullptr);
    int after = block_exclusive_suffix_scan<NT, int>(tmin, MinOp(), INT_MAX, swi);
    int cur = max(before, rs_seed);
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      if (head[i]) cur = base + i;
      rs[i] = cur;
    }
    cur = min(after, re_seed);
#pragma unroll
    for (int i = ITEMS - 1; i >= 0; --i) {
      if (tail[i]) cur = base + i;
      re[i] = cur;
    }
  }

  // Per-thread chunk-head counts packed as (chunks << 32) | long_chunks.
  __device__ long long counts(int n, int s_begin) const {
    const int base = s_begin + threadIdx.x * ITEMS;
    long long c = 0;
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int s = base + i;
      if (s < n && (s - rs[i]) % kNrows == 0) {
        c += 1ll << 32;
        if (re[i] - rs[i] + 1 > kNrows) c += 1;
      }
    }
    return c;
  }

  // Writes the descriptors of the chunks that start in this thread's slots.
  __device__ void emit(const PlanArgs& a, const uint32_t* vals, int s_begin,
                       long long prefix) const {
    const int base = s_begin + threadIdx.x * ITEMS;
    int ci = static_cast<int>(prefix >> 32);
    int lc = static_cast<int>(prefix & 0xffffffffll);
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int s = base + i;
      if (s >= a.n || (s - rs[i]) % kNrows != 0) continue;
      const int L = re[i] - rs[i] + 1;
      const int c = (s - rs[i]) / kNrows;
      const int len = min(kNrows, re[i] - s + 1);
      const bool is_long = L > kNrows;
      int4* d = reinterpret_cast<int4*>(a.chunks + static_cast<long long>(ci) * kChunkWords);
      int p[kNrows];
#pragma unroll
      for (int k = 0; k < kNrows; ++k) p[k] = k < len ? static_cast<int>(vals[s + k]) : 0;
      d[0] = make_int4(p[0], p[1], p[2], p[3]);
      d[1] = make_int4(p[4], p[5], p[6], p[7]);
      d[2] = make_int4(p[8], p[9], static_cast<int>(key[i]), len | (c << 4));
      d[3] = make_int4(is_long ? lc : -1, (L + kNrows - 1) / kNrows, 0, 0);
      if (is_long && c == 0) {
        int* cnt = a.counters + static_cast<long long>(lc) * a.slices;
        for (int j = 0; j < a.slices; ++j) cnt[j] = 0;
      }
      ++ci;
      if (is_long) ++lc;
    }
  }
};

__device__ void write_header(const PlanArgs& a, int chunks, int long_chunks, int bad) {
  Header* h = a.header;
  h->num_chunks = chunks;
  h->num_long_chunks = long_chunks;
  h->bad_ids = bad;
  h->n = a.n;
  h->hidden = a.hidden;
  h->num_embeddings = a.num_embeddings;
  h->status = bad ? EWG_ERR_ID_OUT_OF_RANGE : EWG_OK;
}

// ---------------------------------------------------------------------------
// Single-CTA plan for n <= 8192: keys live in shared memory throughout.

constexpr size_t kSmallSmem =
    static_cast<size_t>(4) * kSmallMaxN * 4 + static_cast<size_t>(1 << kMaxDigitBits) * 32 * 4;

__global__ void __launch_bounds__(kSmallThreads, 1) plan_small_kernel(PlanArgs a) {
  extern __shared__ __align__(16) uint32_t sm[];
  uint32_t* ks = sm;
  uint32_t* vs = ks + kSmallMaxN;
  uint32_t* kd = vs + kSmallMaxN;
  uint32_t* vd = kd + kSmallMaxN;
  uint32_t* cnt = vd + kSmallMaxN;   // [bucket][warp]
  __shared__ long long sw64[32];
  __shared__ int swi[32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  constexpr int NW = kSmallThreads / 32;

  int bad = 0;
#pragma unroll
  for (int r = 0; r < kSmallItems; ++r) {
    const int i = r * kSmallThreads + t;
    ks[i] = make_key(a, i, bad);
    vs[i] = static_cast<uint32_t>(i);
  }
  bad = block_sum_int<kSmallThreads>(bad, sw64);

  for (int pass = 0; pass < a.passes; ++pass) {
    const int sh = pass * a.digit_bits;
    const int bits = min(a.digit_bits, a.id_bits - sh);
    const uint32_t B = 1u << bits, mask = B - 1;
    for (uint32_t i = t; i < B * NW; i += kSmallThreads) cnt[i] = 0;
    __syncthreads();
    uint32_t key[kSmallItems], val[kSmallItems], rank[kSmallItems], dig[kSmallItems];
    // warp w ranks its 256 keys in (round, lane) order, which is input order
#pragma unroll
    for (int r = 0; r < kSmallItems; ++r) {
      const int idx = warp * (32 * kSmallItems) + r * 32 + lane;
      key[r] = ks[idx];
      val[r] = vs[idx];
      const uint32_t d = (key[r] >> sh) & mask;
      const unsigned peers = __match_any_sync(kFull, d);
      const uint32_t below = __popc(peers & ((1u << lane) - 1u));
      const uint32_t prior = cnt[d * NW + warp];
      __syncwarp();
      if (lane == 31 - __clz(peers)) cnt[d * NW + warp] = prior + __popc(peers);
      __syncwarp();
      rank[r] = prior + below;
      dig[r] = d;
    }
    __syncthreads();
    // exclusive scan of cnt in (bucket, warp) order
    {
      const int E = static_cast<int>(B) * NW;
      const int per = (E + kSmallThreads - 1) / kSmallThreads;
      const int b0 = min(E, t * per), b1 = min(E, b0 + per);
      long long local = 0;
      for (int i = b0; i < b1; ++i) local += cnt[i];
      long long run = block_exclusive_scan<kSmallThreads, long long>(local, SumOp(), 0ll, sw64,
                                                                    nullptr);
      for (int i = b0; i < b1; ++i) {
        const uint32_t c = cnt[i];
        cnt[i] = static_cast<uint32_t>(run);
        run += c;
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kSmallItems; ++r) {
      const uint32_t dst = cnt[dig[r] * NW + warp] + rank[r];
      kd[dst] = key[r];
      vd[dst] = val[r];
    }
    __syncthreads();
    uint32_t* tk = ks; ks = kd; kd = tk;
    uint32_t* tv = vs; vs = vd; vd = tv;
  }

  Listing<kSmallThreads, kSmallItems> L;
  L.compute(ks, a.n, 0, 0, a.n - 1, swi);
  long long total = 0;
  long long prefix = block_exclusive_scan<kSmallThreads, long long>(L.counts(a.n, 0), SumOp(),
                                                                   0ll, sw64, &total);
  if (!bad) L.emit(a, vs, 0, prefix);
  if (t == 0) write_header(a, static_cast<int>(total >> 32),
                           static_cast<int>(total & 0xffffffffll), bad);
}

// ---------------------------------------------------------------------------
// Multi-CTA plan: tiles of kTile keys, one CTA each.

// Keys of the tile into the ping buffer, plus the pass-0 digit histogram.
__global__ void __launch_bounds__(kTileThreads) pack_hist_kernel(PlanArgs a) {
  __shared__ uint32_t h[1 << kMaxDigitBits];
  __shared__ long long sw64[kTileThreads / 32];
  const int t = threadIdx.x, tile = blockIdx.x;
  const int B = a.passes ? 1 << min(a.digit_bits, a.id_bits) : 0;
  for (int i = t; i < B; i += kTileThreads) h[i] = 0;
  __syncthreads();
  int bad = 0;
  for (int r = 0; r < kTileItems; ++r) {
    const int i = tile * kTile + r * kTileThreads + t;
    const uint32_t k = make_key(a, i, bad);
    a.keys_a[i] = k;
    a.vals_a[i] = static_cast<uint32_t>(i);
    if (B) atomicAdd(&h[k & (B - 1)], 1u);
  }
  bad = block_sum_int<kTileThreads>(bad, sw64);
  __syncthreads();
  for (int d = t; d < B; d += kTileThreads) a.hist[static_cast<long long>(d) * a.tiles + tile] = h[d];
  if (t == 0) a.tile_bad[tile] = bad;
}

// Digit histogram of each tile for pass >= 1.
__global__ void __launch_bounds__(kTileThreads) hist_kernel(PlanArgs a, const uint32_t* keys,
                                                            int pass) {
  __shared__ uint32_t h[1 << kMaxDigitBits];
  const int t = threadIdx.x, tile = blockIdx.x;
  const int sh = pass * a.digit_bits;
  const int B = 1 << min(a.digit_bits, a.id_bits - sh);
  for (int i = t; i < B; i += kTileThreads) h[i] = 0;
  __syncthreads();
  for (int r = 0; r < kTileItems; ++r) {
    const uint32_t k = keys[tile * kTile + r * kTileThreads + t];
    atomicAdd(&h[(k >> sh) & (B - 1)], 1u);
  }
  __syncthreads();
  for (int d = t; d < B; d += kTileThreads) a.hist[static_cast<long long>(d) * a.tiles + tile] = h[d];
}

// Exclusive scan of hist[bucket][tile] in (bucket, tile) order: each (bucket, tile)
// gets the first output slot of its keys.
__global__ void __launch_bounds__(1024) scan_hist_kernel(PlanArgs a, int pass) {
  __shared__ long long sw64[32];
  const int t = threadIdx.x;
  const int sh = pass * a.digit_bits;
  const long long E = static_cast<long long>(1 << min(a.digit_bits, a.id_bits - sh)) * a.tiles;
  const long long per = (E + 1023) / 1024;
  const long long b0 = min(E, t * per), b1 = min(E, b0 + per);
  long long local = 0;
  for (long long i = b0; i < b1; ++i) local += a.hist[i];
  long long run = block_exclusive_scan<1024, long long>(local, SumOp(), 0ll, sw64, nullptr);
  for (long long i = b0; i < b1; ++i) {
    const uint32_t c = a.hist[i];
    a.hist[i] = static_cast<uint32_t>(run);
    run += c;
  }
}

// Stable scatter of one tile for one pass.
__global__ void __launch_bounds__(kTileThreads) scatter_kernel(PlanArgs a, const uint32_t* ks,
                                                               const uint32_t* vs, uint32_t* kd,
                                                               uint32_t* vd, int pass) {
  constexpr int NW = kTileThreads / 32;
  __shared__ uint32_t cnt[(1 << kMaxDigitBits) * NW];   // [bucket][warp]
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, tile = blockIdx.x;
  const int sh = pass * a.digit_bits;
  const uint32_t B = 1u << min(a.digit_bits, a.id_bits - sh), mask = B - 1;
  for (uint32_t i = t; i < B * NW; i += kTileThreads) cnt[i] = 0;
  __syncthreads();
  uint32_t key[kTileItems], val[kTileItems], rank[kTileItems], dig[kTileItems];
#pragma unroll
  for (int r = 0; r < kTileItems; ++r) {
    const int idx = tile * kTile + warp * (32 * kTileItems) + r * 32 + lane;
    key[r] = ks[idx];
    val[r] = vs[idx];
    const uint32_t d = (key[r] >> sh) & mask;
    const unsigned peers = __match_any_sync(kFull, d);
    const uint32_t below = __popc(peers & ((1u << lane) - 1u));
    const uint32_t prior = cnt[d * NW + warp];
    __syncwarp();
    if (lane == 31 - __clz(peers)) cnt[d * NW + warp] = prior + __popc(peers);
    __syncwarp();
    rank[r] = prior + below;
    dig[r] = d;
  }
  __syncthreads();
  // per bucket: offsets of the warps inside the tile, plus the tile's global base
  for (uint32_t d = t; d < B; d += kTileThreads) {
    uint32_t run = a.hist[static_cast<long long>(d) * a.tiles + tile];
    for (int w = 0; w < NW; ++w) {
      const uint32_t c = cnt[d * NW + w];
      cnt[d * NW + w] = run;
      run += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kTileItems; ++r) {
    const uint32_t dst = cnt[dig[r] * NW + warp] + rank[r];
    kd[dst] = key[r];
    vd[dst] = val[r];
  }
}

// Run bounds of the slots at the two ends of a tile, found by warp 0.
__device__ void tile_seeds(const uint32_t* keys, int n, int s0, int* rs_seed, int* re_seed) {
  __shared__ int seeds[2];
  if (threadIdx.x < 32) {
    const int s1 = min(n, s0 + kTile) - 1;
    const int rs = warp_bound(keys, 0, s0 + 1, keys[s0], false);
    const int re = warp_bound(keys, s1, n, keys[s1], true) - 1;
    if (threadIdx.x == 0) {
      seeds[0] = rs;
      seeds[1] = re;
    }
  }
  __syncthreads();
  *rs_seed = seeds[0];
  *re_seed = seeds[1];
}

__global__ void __launch_bounds__(kTileThreads) list_count_kernel(PlanArgs a,
                                                                  const uint32_t* keys) {
  __shared__ int swi[kTileThreads / 32];
  __shared__ long long sw64[kTileThreads / 32];
  const int s0 = blockIdx.x * kTile;
  int rs_seed, re_seed;
  tile_seeds(keys, a.n, s0, &rs_seed, &re_seed);
  Listing<kTileThreads, kTileItems> L;
  L.compute(keys, a.n, s0, rs_seed, re_seed, swi);
  long long total = 0;
  block_exclusive_scan<kTileThreads, long long>(L.counts(a.n, s0), SumOp(), 0ll, sw64, &total);
  if (threadIdx.x == 0) a.tile_cnt[blockIdx.x] = total;
}

// Scans the per-tile chunk counts, sums the bad-id counts and writes the header.
__global__ void __launch_bounds__(1024) list_scan_kernel(PlanArgs a) {
  __shared__ long long sw64[32];
  const int t = threadIdx.x;
  const int per = (a.tiles + 1023) / 1024;
  const int b0 = min(a.tiles, t * per), b1 = min(a.tiles, b0 + per);
  long long local = 0;
  int bad = 0;
  for (int i = b0; i < b1; ++i) {
    local += a.tile_cnt[i];
    bad += a.tile_bad[i];
  }
  long long total = 0;
  long long run = block_exclusive_scan<1024, long long>(local, SumOp(), 0ll, sw64, &total);
  for (int i = b0; i < b1; ++i) {
    const long long c = a.tile_cnt[i];
    a.tile_cnt[i] = run;
    run += c;
  }
  bad = block_sum_int<1024>(bad, sw64);
  if (t == 0) write_header(a, static_cast<int>(total >> 32), static_cast<int>(total & 0xffffffffll),
                           bad);
}

__global__ void __launch_bounds__(kTileThreads) list_emit_kernel(PlanArgs a, const uint32_t* keys,
                                                                 const uint32_t* vals) {
  __shared__ int swi[kTileThreads / 32];
  __shared__ long long sw64[kTileThreads / 32];
  if (a.header->status != EWG_OK) return;
  const int s0 = blockIdx.x * kTile;
  int rs_seed, re_seed;
  tile_seeds(keys, a.n, s0, &rs_seed, &re_seed);
  Listing<kTileThreads, kTileItems> L;
  L.compute(keys, a.n, s0, rs_seed, re_seed, swi);
  long long prefix = block_exclusive_scan<kTileThreads, long long>(L.counts(a.n, s0), SumOp(), 0ll,
                                                                  sw64, nullptr);
  L.emit(a, vals, s0, prefix + a.tile_cnt[blockIdx.x]);
}

}  // namespace

cudaError_t prepare_plan_kernels() {
  static_assert(kSmallSmem <= 227 * 1024, "single-CTA plan must fit in shared memory");
  return cudaFuncSetAttribute(plan_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmallSmem));
}

cudaError_t launch_plan(const PlanArgs& a, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  if (a.n <= kSmallMaxN) {
    plan_small_kernel<<<1, kSmallThreads, kSmallSmem, stream>>>(a);
    return cudaGetLastError();
  }
  const int tiles = a.tiles;
  pack_hist_kernel<<<tiles, kTileThreads, 0, stream>>>(a);
  const uint32_t* ks = a.keys_a;
  const uint32_t* vs = a.vals_a;
  uint32_t* kd = a.keys_b;
  uint32_t* vd = a.vals_b;
  for (int pass = 0; pass < a.passes; ++pass) {
    if (pass > 0) hist_kernel<<<tiles, kTileThreads, 0, stream>>>(a, ks, pass);
    scan_hist_kernel<<<1, 1024, 0, stream>>>(a, pass);
    scatter_kernel<<<tiles, kTileThreads, 0, stream>>>(a, ks, vs, kd, vd, pass);
    const uint32_t* nk = kd;
    const uint32_t* nv = vd;
    kd = const_cast<uint32_t*>(ks);
    vd = const_cast<uint32_t*>(vs);
    ks = nk;
    vs = nv;
  }
  list_count_kernel<<<tiles, kTileThreads, 0, stream>>>(a, ks);
  list_scan_kernel<<<1, 1024, 0, stream>>>(a);
  list_emit_kernel<<<tiles, kTileThreads, 0, stream>>>(a, ks, vs);
  return cudaGetLastError();
}

}  // namespace ewg
