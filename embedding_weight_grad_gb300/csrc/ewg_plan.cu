// Plan kernels: id validation, (token, position) sort and run / chunk listing.
//
// Counterpart of _sort_tokens_kernel (Megatron Core API docs,
// core.fusions.fused_embedding_wgrad, "Functions"): sort the (token, position) pairs,
// give every sorted slot its run, list the chunks of at most NROWS slots and the runs
// longer than NROWS.
//
// Up to 8192 tokens (hashed path): 64 CTAs each read all ids and keep the ids of one
// hash partition (id * golden-ratio constant, top 6 bits), in position order.  Each
// CTA groups its partition through a shared-memory hash table and ranks every key
// among the earlier keys of its id; a key's chunk and place in the chunk follow from
// its rank, so the pairs are never sorted.  A run never spans two partitions, so no
// CTA waits for another, and the apply kernels find each partition's lists through
// the partition tables.
//
// Above 8192 tokens (multi-tile path): an LSD radix sort over the id bits only (keys
// arrive in position order and every pass is stable, so positions stay ascending in
// each run without passes of their own) over tiles of 2048 keys, one kernel per pass:
// each tile ranks its keys and finds where its digits start from the digit histograms of
// all tiles, which the kernel before it completed (a single sweep per pass, in the
// manner of a "onesweep" radix sort), then one listing kernel that places its chunks by
// decoupled look-back over the tiles before it.
//
// The listing gives every sorted slot s its run's first slot rs and last slot re.
// Slot s starts a chunk when (s - rs) % NROWS == 0.
#include <climits>

#include "ewg.h"
#include "ewg_internal.cuh"
#include "ewg_ptx.cuh"

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
struct SumIntOp {
  __device__ int operator()(int a, int b) const { return a + b; }
};

// Exclusive prefix scan over the block in thread order.  `sw` needs NT/32 entries.
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
    T s = lane < NW ? sw[lane] : ident;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_up_sync(kFull, s, o);
      if (lane >= o) s = op(y, s);
    }
    if (lane < NW) sw[lane] = s;
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
    T s = lane < NW ? sw[lane] : ident;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_down_sync(kFull, s, o);
      if (lane + o < 32) s = op(s, y);
    }
    if (lane < NW) sw[lane] = s;
  }
  __syncthreads();
  T after_warp = warp + 1 < NW ? sw[warp + 1] : ident;
  T down = __shfl_down_sync(kFull, x, 1);
  T excl = op(lane < 31 ? down : ident, after_warp);
  __syncthreads();
  return excl;
}

template <int NT>
__device__ long long block_sum(long long v, long long* sw64) {
  long long tot = 0;
  block_exclusive_scan<NT, long long>(v, SumOp(), 0ll, sw64, &tot);
  return tot;
}

__device__ __forceinline__ long long load_id(const void* ids, int is64, int i) {
  return is64 ? static_cast<const long long*>(ids)[i] : static_cast<const int*>(ids)[i];
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

// Per-thread counts packed in one 64-bit word, 21 bits per field (block-local counts
// stay below 2^21): short chunks << 42 | long chunks << 21 | long runs.
constexpr int kField = 21;
constexpr long long kFieldMask = (1ll << kField) - 1;
__device__ __forceinline__ int field_short(long long p) { return static_cast<int>(p >> (2 * kField)); }
__device__ __forceinline__ int field_long(long long p) { return static_cast<int>((p >> kField) & kFieldMask); }
__device__ __forceinline__ int field_runs(long long p) { return static_cast<int>(p & kFieldMask); }

struct EmitBases {
  int long_desc;     // descriptor index of the first long chunk
  int short_desc;    // descriptor index of the first short chunk
  int partial;       // partial row of the first long chunk
  int run;           // long-run table index of the first long run
};

// Listing of one block of slots [s_begin, s_begin + NT*ITEMS), thread-blocked.
// rs_seed: first slot of the run of slot s_begin; re_seed: last slot of the run of
// the block's last valid slot.
template <int NT, int ITEMS>
struct Listing {
  int rs[ITEMS];
  int re[ITEMS];
  uint32_t key[ITEMS];

  // skey: the keys of slots s_begin - 1 .. s_begin + NT * ITEMS, staged in shared memory.
  __device__ void compute(const uint32_t* skey, int n, int s_begin, int rs_seed, int re_seed,
                          int* swi) {
    const int base = s_begin + threadIdx.x * ITEMS;
    bool head[ITEMS], tail[ITEMS];
    int hmax = -1, tmin = INT_MAX;
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int s = base + i, l = threadIdx.x * ITEMS + i + 1;   // slot s is skey[l]
      head[i] = tail[i] = false;
      key[i] = kPadKey;
      if (s < n) {
        key[i] = skey[l];
        head[i] = (s == 0) || skey[l - 1] != key[i];
        tail[i] = (s == n - 1) || skey[l + 1] != key[i];
        if (head[i]) hmax = max(hmax, s);
        if (tail[i]) tmin = min(tmin, s);
      }
    }
    const int before = block_exclusive_scan<NT, int>(hmax, MaxOp(), -1, swi, nullptr);
    const int after = block_exclusive_suffix_scan<NT, int>(tmin, MinOp(), INT_MAX, swi);
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

  __device__ long long counts(int n, int s_begin, uint32_t skip_key) const {
    const int base = s_begin + threadIdx.x * ITEMS;
    long long c = 0;
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int s = base + i;
      if (s < n && key[i] != skip_key && (s - rs[i]) % kNrows == 0) {
        if (re[i] - rs[i] + 1 > kNrows) {
          c += 1ll << kField;
          if (s == rs[i]) c += fold_entries((re[i] - rs[i] + kNrows) / kNrows);
        } else {
          c += 1ll << (2 * kField);
        }
      }
    }
    return c;
  }

  // Writes the descriptors of the chunks that start in this thread's slots; `prefix`
  // is the packed count of the chunks and runs before this thread's slots.  sval: the
  // positions of slots s_begin .. s_begin + NT * ITEMS + NROWS - 1, staged in shared memory.
  // Each warp's descriptors are contiguous in their list (long chunks, short chunks), so
  // the warp builds them in its shared-memory stage (`wstage`, kEmitStage int4; `wmap`,
  // kEmitMap ints) and writes each list's run of them with coalesced 16-byte stores: one
  // thread's 64-byte descriptors written directly sit 256 bytes apart across the warp,
  // a partial sector per lane.
  static constexpr int kWarpDescs = 32 * ITEMS;        // descriptors of a warp, at most
  static constexpr int kEmitStage = kWarpDescs * kChunkWords / 4;
  static constexpr int kEmitMap = 2 * kWarpDescs;
  __device__ void emit(const PlanArgs& a, const uint32_t* sval, int n, int s_begin,
                       long long prefix, const EmitBases& b, int4* wstage, int* wmap) const {
    const int base = s_begin + threadIdx.x * ITEMS;
    const int lane = static_cast<int>(threadIdx.x & 31);
    int si = field_short(prefix), li = field_long(prefix), ri = field_runs(prefix);
    const int li0 = __shfl_sync(kFull, li, 0), si0 = __shfl_sync(kFull, si, 0);
    int nd = 0;   // this thread's descriptors so far: part q of the nd-th sits at
                  // wstage[(nd * 4 + q) * 32 + (lane ^ q)] (conflict-free both ways)
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int s = base + i;
      if (s >= n || key[i] == a.skip_key || (s - rs[i]) % kNrows != 0) continue;
      const int L = re[i] - rs[i] + 1;
      const int c = (s - rs[i]) / kNrows;
      const int len = min(kNrows, re[i] - s + 1);
      const int C = (L + kNrows - 1) / kNrows;
      const bool is_long = L > kNrows;
      const int desc = is_long ? b.long_desc + li : b.short_desc + si;
      const int prow = is_long ? b.partial + li : -1;
      const bool ok = checked(desc >= 0 && desc < a.chunk_cap && prow < a.partial_cap &&
                                  (!is_long || c != 0 || b.run + ri + fold_entries(C) <= a.run_cap),
                              a.header);
      int p[kNrows];
#pragma unroll
      for (int k = 0; k < kNrows; ++k) {
        p[k] = k < len ? static_cast<int>(sval[s - s_begin + k]) : 0;
        if (!checked(p[k] >= 0 && p[k] < n, a.header)) p[k] = 0;
      }
      wstage[(nd * 4 + 0) * 32 + (lane ^ 0)] = make_int4(p[0], p[1], p[2], p[3]);
      wstage[(nd * 4 + 1) * 32 + (lane ^ 1)] = make_int4(p[4], p[5], p[6], p[7]);
      wstage[(nd * 4 + 2) * 32 + (lane ^ 2)] = make_int4(p[8], p[9], static_cast<int>(key[i]), len | (c << 4));
      wstage[(nd * 4 + 3) * 32 + (lane ^ 3)] = make_int4(prow, C, 0, 0);
      // where the writer finds it: the descriptor's place in the warp's run of its list
      wmap[is_long ? li - li0 : kWarpDescs + si - si0] = ok ? (lane | (nd << 5)) : -1;
      ++nd;
      if (!ok) {   // nothing written for it but its (skipped) place in the list
        if (is_long) ++li;
        else ++si;
        continue;
      }
      if (is_long) {
        if (c == 0) {
          const int split = fold_entries(C);
          for (int q = 0; q < split; ++q)
            reinterpret_cast<int4*>(a.runs)[b.run + ri + q] =
                make_int4(prow, C, static_cast<int>(key[i]), q | (split << 4));
          a.arrivals[prow] = 0;
          ri += split;
        }
        ++li;
      } else {
        ++si;
      }
    }
    __syncwarp();
    const int nl = __shfl_sync(kFull, li, 31) - li0, ns = __shfl_sync(kFull, si, 31) - si0;
    int4* const dst_long = reinterpret_cast<int4*>(a.chunks) + static_cast<long long>(b.long_desc + li0) * 4;
    int4* const dst_short = reinterpret_cast<int4*>(a.chunks) + static_cast<long long>(b.short_desc + si0) * 4;
    for (int q = lane; q < 4 * (nl + ns); q += 32) {
      const int g = q >> 2, part = q & 3;
      const bool lng = g < nl;
      const int m = wmap[lng ? g : kWarpDescs + g - nl];
      if (m < 0) continue;
      const int4 v = wstage[((m >> 5) * 4 + part) * 32 + ((m & 31) ^ part)];
      if (lng) dst_long[q] = v;
      else dst_short[q - 4 * nl] = v;
    }
  }
};

// Everything of the header but its status word: the plan's stamp and the apply kernel's
// counters.
__device__ void write_header_fields(const PlanArgs& a, int num_parts, int bad) {
  Header* h = a.header;
  h->n = a.n;
  h->hidden = a.hidden;
  h->num_embeddings = a.shard_rows;   // rows of the main_grad the apply may touch
  h->num_parts = num_parts;
  h->bad_ids = bad;
  h->work[0] = h->work[1] = 0;
  h->done = 0;
  h->epoch = 0;
  h->spin_limit = kFoldSpinLimit;
}

__device__ void write_header(const PlanArgs& a, int num_parts, int bad) {
  write_header_fields(a, num_parts, bad);
  a.header->status = bad ? EWG_ERR_ID_OUT_OF_RANGE : EWG_OK;
}

__device__ void write_tables(const PlanArgs& a, int part, int long_cnt, int long_off,
                             int short_cnt, int short_off, int run_cnt, int run_off) {
  a.tables[kLongCnt * kMaxParts + part] = long_cnt;
  a.tables[kLongOff * kMaxParts + part] = long_off;
  a.tables[kShortCnt * kMaxParts + part] = short_cnt;
  a.tables[kShortOff * kMaxParts + part] = short_off;
  a.tables[kRunCnt * kMaxParts + part] = run_cnt;
  a.tables[kRunOff * kMaxParts + part] = run_off;
}

__device__ __forceinline__ int hash_part(uint32_t id) {
  static_assert(kHashParts == 64, "hash uses the top 6 bits");
  return static_cast<int>((id * 0x9E3779B1u) >> 26);
}

// Slot hash of the per-partition table, independent of the partition hash.
__device__ __forceinline__ uint32_t hash_slot(uint32_t id, int tbits) {
  return (id * 0x85EBCA77u) >> (32 - tbits);
}

constexpr int kHashWarps = kHashThreads / 32;
constexpr int kTableMax = kHashMaxN;           // table slots at most (a power of two)
constexpr uint32_t kEmptySlot = 0xffffffffu;
constexpr int kRankShift = 13;                 // key info word: slot | rank << 13
constexpr uint32_t kSlotMask = (1u << kRankShift) - 1u;
// key info word between the probe and the ranks: slot | rank in the 32-key group |
// lane of the group's last key of the id | that id's keys in the group - 1
constexpr int kInRankShift = 13, kLastShift = 18, kGroupCntShift = 23;
static_assert(kTableMax <= (1 << kRankShift) && kHashMaxN <= (1 << (32 - kRankShift)),
              "slot and rank must pack into one word");
constexpr size_t kHashSmem =
    static_cast<size_t>(2) * kHashMaxN * 4 + static_cast<size_t>(4) * kTableMax * 4;
constexpr int kListWarps = kHashWarps - 1;     // warps that list the runs while warp 0 ranks

// Exclusive sum over the threads of warps 1..kListWarps of the block, synchronised by
// named barrier 1 (warp 0 does other work meanwhile); *total = the sum over all of them.
__device__ long long list_warps_exclusive_sum(long long v, long long* sw, long long* total) {
  const int lane = threadIdx.x & 31, w = static_cast<int>(threadIdx.x >> 5) - 1;
  constexpr int kCount = kListWarps * 32;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sw[w] = x;
  asm volatile("bar.sync 1, %0;" ::"n"(kCount) : "memory");
  if (w == 0) {
    long long q = lane < kListWarps ? sw[lane] : 0ll;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(kFull, q, o);
      if (lane >= o) q += y;
    }
    if (lane < kListWarps) sw[lane] = q;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kCount) : "memory");
  const long long before_warp = w > 0 ? sw[w - 1] : 0ll;
  const long long up = __shfl_up_sync(kFull, x, 1);
  *total = sw[kListWarps - 1];
  return before_warp + (lane > 0 ? up : 0ll);
}

// ---------------------------------------------------------------------------
// Hashed plan: CTA `part` handles the ids whose hash partition is `part`.
//
// Inside the partition a shared-memory hash table gives every distinct id a slot.  One
// warp then walks the keys in position order, 32 at a time, and gives each key its
// rank among the earlier keys of its id (match.any groups equal slots within the 32).
// A key's chunk is rank / NROWS and its place in the chunk is rank % NROWS, so the
// (token, position) pairs never need to be sorted: after a scan over the table assigns
// every run its descriptors, every key writes its own position word.

__global__ void __launch_bounds__(kHashThreads, 1) plan_hashed_kernel(PlanArgs a) {
  ptx::pdl_wait_prior_grid();
  ptx::pdl_launch_dependents();
  extern __shared__ __align__(16) uint32_t sm[];
  uint32_t* kpos = sm;                   // position of key i (keys in position order)
  uint32_t* kinfo = kpos + kHashMaxN;    // id of key i; then slot | rank << kRankShift
  uint32_t* tkey = kinfo + kHashMaxN;    // table: id of the slot
  uint32_t* tcnt = tkey + kTableMax;     // table: occurrences of the id (run length)
  uint32_t* tbase = tcnt + kTableMax;    // table: descriptor of the run's first chunk
  uint32_t* wcnt = tbase + kTableMax;    // table: the id's keys ranked so far
  __shared__ int wc[kHashItems * kHashWarps];
  __shared__ long long sw64[kHashWarps];
  __shared__ int s_counts[3];   // long chunks, short chunks, long-run entries
  __shared__ long long s_red;   // bad ids << 32 | tokens of lower partitions
  __shared__ int s_m;           // keys of this partition
  const int part = blockIdx.x;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t lt = (1u << lane) - 1u;

  // 1. every id, striped: round r covers positions [r*NT, (r+1)*NT).  All loads are
  // issued before any is used, so they overlap.
  long long raw[kHashItems];
#pragma unroll
  for (int r = 0; r < kHashItems; ++r) {
    const int p = r * kHashThreads + t;
    raw[r] = p < a.n ? load_id(a.ids, a.ids_int64, p) : 0;
  }
  uint32_t key[kHashItems];
  unsigned ballot[kHashItems];
  int bad = 0, before = 0;
#pragma unroll
  for (int r = 0; r < kHashItems; ++r) {
    const int p = r * kHashThreads + t;
    bool mine = false;
    key[r] = 0;
    if (p < a.n) {
      if (raw[r] < 0 || raw[r] >= a.num_embeddings) {
        ++bad;
      } else if (raw[r] >= a.row_begin && raw[r] - a.row_begin < a.shard_rows) {
        key[r] = static_cast<uint32_t>(raw[r] - a.row_begin);
        const int h = hash_part(key[r]);
        mine = h == part;
        before += h < part;
      }
    }
    ballot[r] = __ballot_sync(kFull, mine);
    if (lane == 0) wc[r * kHashWarps + warp] = __popc(ballot[r]);
  }
  // One pass of warp 0 over the warps' results gives the block's bad ids and tokens of
  // lower partitions, and turns the (round, warp) key counts into offsets in that order
  // (position order) and their total m.
  {
    long long bb = (static_cast<long long>(bad) << 32) | before;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bb += __shfl_xor_sync(kFull, bb, o);
    if (lane == 0) sw64[warp] = bb;
  }
  __syncthreads();
  if (warp == 0) {
    static_assert(kHashWarps == 32 && kHashItems * kHashWarps == 8 * 32, "one lane per warp, 8 counts each");
    long long tot = sw64[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(kFull, tot, o);
    int v[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int x = wc[8 * lane + j];
      v[j] = sum;
      sum += x;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) wc[8 * lane + j] = v[j] + incl - sum;
    if (lane == 31) s_m = incl;
    if (lane == 0) s_red = tot;
  }
  __syncthreads();
  const long long red = s_red;
  const int bad_total = static_cast<int>(red >> 32);
  const int S_b = static_cast<int>(red & 0xffffffffll);   // tokens of partitions < part
  if (bad_total) {
    if (part == 0 && t == 0) write_header(a, kHashParts, bad_total);
    return;
  }

  // 2. this partition's keys, compacted in position order
  const int m = s_m;
#pragma unroll
  for (int r = 0; r < kHashItems; ++r) {
    if ((ballot[r] >> lane) & 1u) {
      const int i = wc[r * kHashWarps + warp] + __popc(ballot[r] & lt);
      kpos[i] = static_cast<uint32_t>(r * kHashThreads + t);
      kinfo[i] = key[r];
    }
  }
  int tbits = 5;   // table of at least 2m slots (at least m, kTableMax >= every m)
  while ((1 << tbits) < 2 * m && (1 << tbits) < kTableMax) ++tbits;
  const int TS = 1 << tbits;
  for (int s = t; s < TS; s += kHashThreads) {
    tkey[s] = kEmptySlot;
    tcnt[s] = 0;
    wcnt[s] = 0;
  }
  __syncthreads();

  // 3. the slot of every key: linear probing; there are at least as many slots as ids,
  // so every probe sequence ends within TS steps.  Within a warp only one lane per
  // distinct id probes (a hot id would otherwise serialise on one slot) and adds the
  // group's keys to the id's count.
  for (int i0 = warp * 32; i0 < m; i0 += kHashThreads) {
    const int i = i0 + lane;
    const bool valid = i < m;
    const uint32_t id = valid ? kinfo[i] : kEmptySlot;
    const unsigned peers = __match_any_sync(kFull, id);
    const int leader = __ffs(peers) - 1;
    uint32_t h = 0;
    if (valid && lane == leader) {
      h = hash_slot(id, tbits);
      for (int probe = 0; probe < TS; ++probe) {
        const uint32_t cur = tkey[h];
        if (cur == id) break;
        if (cur == kEmptySlot) {
          const uint32_t old = atomicCAS(&tkey[h], kEmptySlot, id);
          if (old == kEmptySlot || old == id) break;
        }
        h = (h + 1) & static_cast<uint32_t>(TS - 1);
      }
      atomicAdd(&tcnt[h], static_cast<uint32_t>(__popc(peers)));   // the id's run length
    }
    h = __shfl_sync(kFull, h, leader);
    // the key's rank among its group's keys of the same id, the group's last such key
    // and their number
    if (valid)
      kinfo[i] = h | (static_cast<uint32_t>(__popc(peers & lt)) << kInRankShift) |
                 (static_cast<uint32_t>(31 - __clz(peers)) << kLastShift) |
                 (static_cast<uint32_t>(__popc(peers) - 1) << kGroupCntShift);
  }
  __syncthreads();

  // 4 and 5 side by side.  Warp 0 gives every key its rank in position order: it carries
  // the per-slot counts across the 32-key groups in order, each group's last key of an id
  // adding the group's count.  Meanwhile the other warps list the runs (their lengths are
  // the probe's counts): a scan over the table gives each run its first descriptor, and
  // long runs also get their partial rows and their row of the long-run table.
  if (warp == 0) {
    uint32_t next = lane < m ? kinfo[lane] : 0u;
    for (int i0 = 0; i0 < m; i0 += 32) {
      const int i = i0 + lane;
      const bool valid = i < m;
      const uint32_t info = next;
      next = i + 32 < m ? kinfo[i + 32] : 0u;
      const uint32_t s = info & kSlotMask;
      const int last = static_cast<int>((info >> kLastShift) & 31u);
      uint32_t prior = 0;
      if (valid && lane == last) {
        prior = wcnt[s];
        wcnt[s] = prior + ((info >> kGroupCntShift) & 31u) + 1u;
      }
      __syncwarp();
      const uint32_t base = __shfl_sync(kFull, prior, last);
      if (valid) kinfo[i] = s | ((base + ((info >> kInRankShift) & 31u)) << kRankShift);
    }
  } else {
    constexpr int NL = kListWarps * 32;
    const int u = t - 32;
    long long cnt = 0;
    for (int s = u; s < TS; s += NL) {
      const int L = static_cast<int>(tcnt[s]);
      if (L > kNrows) {
        const int C = (L + kNrows - 1) / kNrows;
        cnt += (static_cast<long long>(C) << kField) + fold_entries(C);
      } else if (L > 0) {
        cnt += 1ll << (2 * kField);
      }
    }
    long long tot = 0;
    const long long pre = list_warps_exclusive_sum(cnt, sw64, &tot);
    const int n_long = field_long(tot);
    if (u == 0) {
      s_counts[0] = n_long;
      s_counts[1] = field_short(tot);
      s_counts[2] = field_runs(tot);
    }
    const int long_desc = S_b, short_desc = S_b + n_long;
    const int partial_base = (2 * S_b) / 11 + part, run_base = S_b / 11 + S_b / 100 + part;
    int li = field_long(pre), si = field_short(pre), ri = field_runs(pre);
    for (int s = u; s < TS; s += NL) {
      const int L = static_cast<int>(tcnt[s]);
      if (L > kNrows) {
        const int C = (L + kNrows - 1) / kNrows;
        tbase[s] = static_cast<uint32_t>(long_desc + li);
        const int split = fold_entries(C);
        if (checked(run_base + ri + split <= a.run_cap && partial_base + li + C <= a.partial_cap, a.header)) {
          for (int q = 0; q < split; ++q)
            reinterpret_cast<int4*>(a.runs)[run_base + ri + q] =
                make_int4(partial_base + li, C, static_cast<int>(tkey[s]), q | (split << 4));
          a.arrivals[partial_base + li] = 0;
        }
        li += C;
        ri += split;
      } else if (L > 0) {
        tbase[s] = static_cast<uint32_t>(short_desc + si);
        ++si;
      }
    }
  }
  __syncthreads();
  const int n_long = s_counts[0], n_short = s_counts[1], n_runs = s_counts[2];
  const int long_desc = S_b, short_desc = S_b + n_long;
  const int partial_base = (2 * S_b) / 11 + part, run_base = S_b / 11 + S_b / 100 + part;

  // 6. every key writes its position into its chunk; the first key of a chunk also
  // writes the chunk's id, length, index in the run, partial row and the run's size
  for (int i = t; i < m; i += kHashThreads) {
    const uint32_t info = kinfo[i];
    const int s = static_cast<int>(info & ((1u << kRankShift) - 1u));
    const int r = static_cast<int>(info >> kRankShift);
    const int L = static_cast<int>(tcnt[s]);
    const int c = r / kNrows, k = r - c * kNrows;
    const int desc = static_cast<int>(tbase[s]) + c;
    if (!checked(desc >= 0 && desc < a.chunk_cap && kpos[i] < static_cast<uint32_t>(a.n), a.header)) continue;
    int* d = a.chunks + static_cast<long long>(desc) * kChunkWords;
    d[kDescPos + k] = static_cast<int>(kpos[i]);
    if (k == 0) {
      const bool is_long = L > kNrows;
      const int len = min(kNrows, L - r);
      const int C = (L + kNrows - 1) / kNrows;
      const int prow = is_long ? partial_base + (static_cast<int>(tbase[s]) - long_desc) + c : -1;
      reinterpret_cast<int2*>(d)[kDescId / 2] = make_int2(static_cast<int>(tkey[s]), len | (c << 4));
      reinterpret_cast<int4*>(d)[kDescPartial / 4] = make_int4(prow, C, 0, 0);
    }
  }
  if (t == 0) {
    write_tables(a, part, n_long, long_desc, n_short, short_desc, n_runs, run_base);
    if (part == 0) write_header(a, kHashParts, 0);
  }
}

// ---------------------------------------------------------------------------
// Multi-tile plan: tiles of kTile keys, one CTA each.
//
//   pack    each tile's keys (the id, or a skip / pad key) and positions, its bad ids and
//           its digit histogram for the first radix pass; clears what later kernels count
//           into
//   sweep   one per radix pass: a stable scatter.  Each tile sums the histogram columns
//           of its digits over all tiles (keys of smaller digits come first) and over the
//           tiles before it (its own keys of a digit follow theirs), ranks its keys and
//           scatters them; it also counts, per destination tile, the digits of the next
//           pass, so the next sweep finds its histograms complete.  No tile waits for
//           another.
//   list    runs and chunks of the sorted keys: each tile counts its chunks and runs,
//           sums the counts of the tiles before it by decoupled look-back (tiles are taken
//           in claim order, so the tiles before a running one are running or done, and
//           every poll is bounded), and writes its descriptors; the last tile writes the
//           tables and the header.
// A look-back that gives up sets EWG_ERR_TIMEOUT and the tile writes nothing.
//
// Each sweep reads the histograms of all tiles for its digits: tiles x 2 KB per CTA, one
// round of loads up to a few hundred tiles, growing with the square of the tile count
// beyond.

constexpr uint32_t kFlagAgg = 1u << 30;   // the word holds the tile's own count
constexpr uint32_t kFlagInc = 2u << 30;   // ... the sum over the tile and all before it
constexpr uint32_t kCountMask = kFlagAgg - 1u;
constexpr int kLookBackPolls = 1 << 20;   // poll rounds of one look-back (about 0.5 s)

__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Decoupled look-back by one whole warp over one chain of words (tile j's word at word +
// j * stride).  The tile has already published its own count (as tile 0, an inclusive
// sum).  Each round loads the words of the up to 32 closest predecessors not yet summed,
// one per lane, all in flight together; re-polls together the ones not yet published
// before the closest inclusive word; then adds by a warp reduction the counts from the
// closest predecessor back to that inclusive word, or all of them when there is none and
// the next 32 follow.  So each round costs one or two round trips whatever the number of
// predecessors.  Publishes this tile's inclusive sum and gives every lane the exclusive
// sum in *excl.  False (nothing published) if a predecessor published nothing within
// poll_limit polls.
__device__ bool warp_look_back(uint32_t* word, long long stride, int tile, uint32_t own, uint32_t* excl,
                               int poll_limit = kLookBackPolls) {
  const int lane = static_cast<int>(threadIdx.x & 31);
  uint32_t sum = 0;
  for (int hi = tile; hi > 0;) {
    const int m = min(hi, 32);
    const bool valid = lane < m;
    uint32_t* w = word + static_cast<long long>(valid ? hi - 1 - lane : hi - 1) * stride;
    uint32_t v = valid ? ld_relaxed(w) : kFlagAgg;   // a lane past the predecessors: count 0
    unsigned inc, need;   // lanes holding inclusive sums; lanes up to the closest of them
    for (int poll = 0;; ++poll) {
      inc = __ballot_sync(kFull, (v & kFlagInc) != 0);
      const unsigned unpub = __ballot_sync(kFull, (v & ~kCountMask) == 0);
      need = inc ? (inc & (0u - inc)) * 2u - 1u : kFull;
      if (!(unpub & need)) break;
      if (poll >= poll_limit) return false;
      __nanosleep(32);
      if ((unpub & need) >> lane & 1u) v = ld_relaxed(w);
    }
    uint32_t x = (need >> lane & 1u) ? (v & kCountMask) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    sum += x;
    if (inc) break;   // the closest inclusive word ended the sum
    hi -= m;
  }
  if (lane == 0) st_relaxed(word + static_cast<long long>(tile) * stride, kFlagInc | (sum + own));
  *excl = sum;
  return true;
}

__device__ void give_up_plan(const PlanArgs& a) { atomicExch(&a.header->status, kStatusTimeout); }

#ifdef EWG_DEBUG
// Test probe of the look-back (bounds-checking build only): one warp looks back from
// `tile` over words prepared by the caller, a word of 0 being a predecessor that never
// publishes, with at most poll_limit polls.  out[0]: 1 if it completed, 0 if it gave up;
// out[1]: the exclusive sum it found.
__global__ void lookback_probe_kernel(uint32_t* words, int tile, int poll_limit, int* out) {
  uint32_t before = 0;
  const bool ok = warp_look_back(words, 1, tile, 1u, &before, poll_limit);
  if (threadIdx.x == 0) {
    out[0] = ok ? 1 : 0;
    out[1] = static_cast<int>(before);
  }
}
#endif

// Digit width of `pass` (the last pass may take fewer bits).
__device__ __forceinline__ uint32_t pass_buckets(const PlanArgs& a, int pass) {
  return 1u << min(a.digit_bits, a.id_bits - pass * a.digit_bits);
}

// The packing takes a tile of kTile ids on kPackThreads threads, kPackItems each.
constexpr int kPackThreads = 1024;
constexpr int kPackItems = kTile / kPackThreads;

__global__ void __launch_bounds__(kPackThreads) pack_kernel(PlanArgs a) {
  constexpr int B = 1 << kMaxDigitBits;
  __shared__ long long sw64[kPackThreads / 32];
  __shared__ uint32_t h[B];
  const int t = threadIdx.x, lane = t & 31, tile = blockIdx.x;
  for (int d = t; d < B; d += kPackThreads) h[d] = 0;
  ptx::pdl_wait_prior_grid();
  ptx::pdl_launch_dependents();
  int bad = 0;
  long long raw[kPackItems];
#pragma unroll
  for (int r = 0; r < kPackItems; ++r) {
    const int i = tile * kTile + r * kPackThreads + t;
    raw[r] = i < a.n ? load_id(a.ids, a.ids_int64, i) : 0;
  }
  __syncthreads();   // h is clear
  const uint32_t mask0 = a.passes ? pass_buckets(a, 0) - 1u : 0u;
#pragma unroll
  for (int r = 0; r < kPackItems; ++r) {
    const int i = tile * kTile + r * kPackThreads + t;
    uint32_t k = kPadKey;
    if (i < a.n) {
      if (raw[r] < 0 || raw[r] >= a.num_embeddings) {
        ++bad;
        k = 0u;
      } else if (raw[r] >= a.row_begin && raw[r] - a.row_begin < a.shard_rows) {
        k = static_cast<uint32_t>(raw[r] - a.row_begin);
      } else {
        k = a.skip_key;   // outside the shard: sorts after its rows, listed as nothing
      }
    }
    a.keys_a[i] = k;
    a.vals_a[i] = static_cast<uint32_t>(i);
    if (a.passes) {   // one atomic per distinct digit per warp: a hot id would serialise
      const uint32_t d = k & mask0;
      const unsigned peers = __match_any_sync(kFull, d);
      if (lane == __ffs(peers) - 1) atomicAdd(&h[d], static_cast<uint32_t>(__popc(peers)));
    }
  }
  bad = static_cast<int>(block_sum<kPackThreads>(bad, sw64));   // its barriers also complete h
  if (t == 0) a.tile_bad[tile] = bad;
  // this tile's histogram of the first pass; its rows of the later passes start at zero
  // (the sweep before each of them counts into them)
  for (int p = 0; p < a.passes; ++p) {
    const int Bp = static_cast<int>(pass_buckets(a, p));
    uint32_t* row = a.tile_hist + (static_cast<long long>(p) * a.tiles + tile) * B;
    for (int d = t; d < Bp; d += kPackThreads) row[d] = p == 0 ? h[d] : 0u;
  }
  if (t < 3) a.list_status[static_cast<long long>(tile) * kStatusWords + t] = 0;
  if (tile == 0) {
    if (t <= kMaxPasses) a.counters[t] = 0;
    if (t == 0) a.header->status = EWG_OK;
  }
}

// The sweep takes a tile of kTile keys on kSweepThreads threads, kSweepItems each; each
// thread owns one digit of the histogram.
constexpr int kSweepThreads = 1 << kMaxDigitBits;
constexpr int kSweepItems = kTile / kSweepThreads;

// One stable LSD radix pass: (ks, vs) -> (kd, vd), ordered by the digit of `pass`.
__global__ void __launch_bounds__(kSweepThreads) sweep_kernel(PlanArgs a, const uint32_t* ks,
                                                              const uint32_t* vs, uint32_t* kd,
                                                              uint32_t* vd, int pass) {
  constexpr int NW = kSweepThreads / 32;
  constexpr int kStride = 1 << kMaxDigitBits;
  constexpr int kBatch = 32;                      // histogram rows loaded together
  static_assert(kStride == kSweepThreads, "each thread owns one digit");
  __shared__ uint32_t cnt[NW * kStride];          // [warp][digit]
  __shared__ uint32_t base[kStride];              // first output slot of the tile's digit
  __shared__ int sw[NW];
  __shared__ int s_ok;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, tile = blockIdx.x;
  const int sh = pass * a.digit_bits;
  const uint32_t B = pass_buckets(a, pass), mask = B - 1;
  const uint32_t lt = (1u << lane) - 1u;
  for (int w = 0; w < NW; ++w)
    if (static_cast<uint32_t>(t) < B) cnt[w * kStride + t] = 0;
  ptx::pdl_wait_prior_grid();
  ptx::pdl_launch_dependents();
  if (t == 0) s_ok = a.header->status == EWG_OK;
  uint32_t key[kSweepItems], val[kSweepItems];
#pragma unroll
  for (int r = 0; r < kSweepItems; ++r) {
    const int idx = tile * kTile + warp * (32 * kSweepItems) + r * 32 + lane;
    key[r] = ks[idx];
    val[r] = vs[idx];
  }
  // this thread's digit d: keys of it over all tiles (tot) and over the tiles before this
  // one (pre), from the complete tile histograms of this pass
  const int d = t;
  const uint32_t* hist = a.tile_hist + static_cast<long long>(pass) * a.tiles * kStride + d;
  uint32_t tot = 0, pre = 0;
  if (static_cast<uint32_t>(d) < B) {
    for (int j0 = 0; j0 < a.tiles; j0 += kBatch) {
      uint32_t v[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        v[i] = j0 + i < a.tiles ? hist[static_cast<long long>(j0 + i) * kStride] : 0u;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        tot += v[i];
        if (j0 + i < tile) pre += v[i];
      }
    }
  }
  __syncthreads();
  if (!s_ok) return;
  uint32_t rank[kSweepItems], dig[kSweepItems];
#pragma unroll
  for (int r = 0; r < kSweepItems; ++r) {
    const uint32_t dd = (key[r] >> sh) & mask;
    const unsigned peers = __match_any_sync(kFull, dd);
    const uint32_t prior = cnt[warp * kStride + dd];
    __syncwarp();
    if (lane == 31 - __clz(peers)) cnt[warp * kStride + dd] = prior + __popc(peers);
    __syncwarp();
    rank[r] = prior + __popc(peers & lt);
    dig[r] = dd;
  }
  // keys of smaller digits over all tiles: an exclusive scan of the totals over the block
  // (its barriers also complete the ranks in cnt), then cnt -> per-warp offsets in the tile
  const int below = block_exclusive_scan<kSweepThreads, int>(static_cast<int>(tot), SumIntOp(), 0, sw, nullptr);
  if (static_cast<uint32_t>(d) < B) {
    uint32_t run = 0;
    for (int w = 0; w < NW; ++w) {
      const uint32_t c = cnt[w * kStride + d];
      cnt[w * kStride + d] = run;
      run += c;
    }
    base[d] = static_cast<uint32_t>(below) + pre;
  }
  __syncthreads();
  const bool next = pass + 1 < a.passes;
  const int nsh = (pass + 1) * a.digit_bits;
  const uint32_t nmask = next ? pass_buckets(a, pass + 1) - 1u : 0u;
  uint32_t* nhist = a.tile_hist + static_cast<long long>(pass + 1) * a.tiles * kStride;
#pragma unroll
  for (int r = 0; r < kSweepItems; ++r) {
    const uint32_t dst = base[dig[r]] + cnt[warp * kStride + dig[r]] + rank[r];
    const bool in = checked(dst < static_cast<uint32_t>(a.tiles) * kTile, a.header);
    if (in) {
      kd[dst] = key[r];
      vd[dst] = val[r];
    }
    if (next) {   // the next pass's digit of this key, in the tile it now belongs to
      const uint32_t slot = in ? (dst / kTile) * kStride + ((key[r] >> nsh) & nmask) : 0u;
      const unsigned peers = __match_any_sync(kFull, slot);
      if (in && lane == __ffs(peers) - 1) atomicAdd(&nhist[slot], static_cast<uint32_t>(__popc(peers)));
    }
  }
}

// Bound of key k, like warp_bound, looking first at the 32 slots next to `at` (the
// start of the search for an upper bound, the end for a lower bound): most runs are
// short, so one load usually settles it.
__device__ int warp_bound_near(const uint32_t* keys, int lo, int hi, int at, uint32_t k, bool upper) {
  const int lane = threadIdx.x & 31;
  if (upper) {   // first index in [at, hi) with key > k
    const int w1 = min(hi, at + 32);
    const int idx = at + lane;
    const bool pred = idx < w1 ? keys[idx] > k : true;
    const unsigned m = __ballot_sync(kFull, pred);
    const int f = __ffs(m) - 1;   // -1 when all 32 slots of a full window hold k
    if (m != 0 && (at + f < w1 || w1 == hi)) return min(at + f, hi);
    return warp_bound(keys, w1, hi, k, true);
  }
  // first index in [lo, at + 1) with key >= k
  const int w0 = max(lo, at - 31);
  const int idx = w0 + lane;
  const bool pred = idx <= at ? keys[idx] >= k : true;
  const unsigned m = __ballot_sync(kFull, pred);
  const int f = __ffs(m) - 1;     // m != 0: slot `at` holds k
  if (f > 0 || w0 == lo) return w0 + f;
  return warp_bound(keys, lo, w0 + 1, k, false);
}

// Run bounds of the slots at the two ends of a tile: warp 0 finds where the run of the
// first slot starts, warp 1 where the run of the last slot ends.
__device__ void tile_seeds(const uint32_t* keys, int n, int s0, int* rs_seed, int* re_seed) {
  __shared__ int seeds[2];
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    const int rs = warp_bound_near(keys, 0, s0 + 1, s0, keys[s0], false);
    if (threadIdx.x == 0) seeds[0] = rs;
  } else if (warp == 1) {
    const int s1 = min(n, s0 + kTile) - 1;
    const int re = warp_bound_near(keys, s1, n, s1, keys[s1], true) - 1;
    if (threadIdx.x == 32) seeds[1] = re;
  }
  __syncthreads();
  *rs_seed = seeds[0];
  *re_seed = seeds[1];
}

// The listing takes a tile of kTile sorted slots on kListThreads threads, kListItems each.
constexpr int kListThreads = 512;
constexpr int kListItems = kTile / kListThreads;

// Runs and chunks of the sorted keys, one tile per CTA (tiles in claim order).  The tile's
// keys (with one slot on each side) and positions (with the NROWS - 1 slots after it) are
// staged in shared memory by one coalesced load.
using ListTile = Listing<kListThreads, kListItems>;
// per warp: the descriptors it builds (transposed) and where its writers find them
constexpr size_t kListDynSmem = static_cast<size_t>(kListThreads / 32) *
                                (ListTile::kEmitStage * sizeof(int4) + ListTile::kEmitMap * sizeof(int));

__global__ void __launch_bounds__(kListThreads) list_kernel(PlanArgs a, const uint32_t* keys,
                                                            const uint32_t* vals) {
  extern __shared__ __align__(16) int4 emit_smem[];   // kListDynSmem
  __shared__ uint32_t skey[kTile + 2];
  __shared__ uint32_t sval[kTile + kNrows];
  __shared__ int swi[kListThreads / 32];
  __shared__ long long sw64[kListThreads / 32];
  __shared__ int s_tile, s_ok;
  __shared__ uint32_t s_before[3], s_own[3];
  const int t = threadIdx.x;
  const long long n_pad = static_cast<long long>(a.tiles) * kTile;
  ptx::pdl_wait_prior_grid();
  ptx::pdl_launch_dependents();
  if (t == 0) {
    s_ok = a.header->status == EWG_OK;
    s_tile = atomicAdd(&a.counters[kMaxPasses], 1);
  }
  long long bad = 0;
  for (int i = t; i < a.tiles; i += kListThreads) bad += a.tile_bad[i];
  __syncthreads();
  if (!s_ok) return;
  const int tile = s_tile;
  const int s0 = tile * kTile;
  {   // every load in flight at once: the tile body as 16-byte vectors, then the halos
    static_assert(kListItems == 4, "one 16-byte vector per thread");
    const uint4 k0 = reinterpret_cast<const uint4*>(keys + s0)[t];
    const uint4 v0 = reinterpret_cast<const uint4*>(vals + s0)[t];
    uint32_t halo = 0u;
    if (t == 0) halo = s0 > 0 ? keys[s0 - 1] : kPadKey;
    else if (t == 1) halo = s0 + kTile < n_pad ? keys[s0 + kTile] : kPadKey;
    else if (t < 2 + kNrows) halo = s0 + kTile + (t - 2) < n_pad ? vals[s0 + kTile + (t - 2)] : 0u;
    uint32_t* sk = skey + 1 + 4 * t;
    uint32_t* sv = sval + 4 * t;
    sk[0] = k0.x, sk[1] = k0.y, sk[2] = k0.z, sk[3] = k0.w;
    sv[0] = v0.x, sv[1] = v0.y, sv[2] = v0.z, sv[3] = v0.w;
    if (t == 0) skey[0] = halo;
    else if (t == 1) skey[kTile + 1] = halo;
    else if (t < 2 + kNrows) sval[kTile + (t - 2)] = halo;
  }
  bad = block_sum<kListThreads>(bad, sw64);   // its barriers also complete the staging
  if (bad) {   // nothing is listed; the first tile reports the bad ids
    if (tile == 0 && t == 0) {
      write_header_fields(a, 1, static_cast<int>(bad));
      atomicExch(&a.header->status, EWG_ERR_ID_OUT_OF_RANGE);
    }
    return;
  }
  int rs_seed, re_seed;
  tile_seeds(keys, a.n, s0, &rs_seed, &re_seed);
  ListTile L;
  L.compute(skey, a.n, s0, rs_seed, re_seed, swi);
  long long tot = 0;
  const long long prefix = block_exclusive_scan<kListThreads, long long>(L.counts(a.n, s0, a.skip_key),
                                                                         SumOp(), 0ll, sw64, &tot);
  if (t < 3 * 32) {   // one look-back chain per warp: long chunks, short chunks, long-run entries
    const int c = t >> 5;
    const uint32_t own = static_cast<uint32_t>(c == 0 ? field_long(tot) : c == 1 ? field_short(tot) : field_runs(tot));
    uint32_t* word = a.list_status + c;
    if ((t & 31) == 0) st_relaxed(word + static_cast<long long>(tile) * kStatusWords, (tile ? kFlagAgg : kFlagInc) | own);
    uint32_t before = 0;
    const bool ok = tile == 0 || warp_look_back(word, kStatusWords, tile, own, &before);
    if ((t & 31) == 0) {
      s_before[c] = ok ? before : 0xffffffffu;
      s_own[c] = own;
    }
  }
  __syncthreads();
  if (s_before[0] == 0xffffffffu || s_before[1] == 0xffffffffu || s_before[2] == 0xffffffffu) {
    if (t == 0) give_up_plan(a);
    return;
  }
  EmitBases eb;
  eb.long_desc = static_cast<int>(s_before[0]);
  eb.short_desc = a.short_base + static_cast<int>(s_before[1]);
  eb.partial = static_cast<int>(s_before[0]);
  eb.run = static_cast<int>(s_before[2]);
  {
    const int w = t >> 5;
    int4* wstage = emit_smem + w * ListTile::kEmitStage;
    int* wmap = reinterpret_cast<int*>(emit_smem + (kListThreads / 32) * ListTile::kEmitStage) +
                w * ListTile::kEmitMap;
    L.emit(a, sval, a.n, s0, prefix, eb, wstage, wmap);
  }
  if (tile == a.tiles - 1 && t == 0) {
    write_tables(a, 0, static_cast<int>(s_before[0] + s_own[0]), 0, static_cast<int>(s_before[1] + s_own[1]),
                 a.short_base, static_cast<int>(s_before[2] + s_own[2]), 0);
    write_header_fields(a, 1, 0);
  }
}

}  // namespace

cudaError_t prepare_kernels() {
  static_assert(kHashSmem <= 227 * 1024, "hashed plan must fit in shared memory");
  static_assert(kListDynSmem + 24 * 1024 <= 227 * 1024, "listing stages must fit in shared memory");
  cudaError_t e = cudaFuncSetAttribute(plan_hashed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kHashSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(list_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kListDynSmem));
}

namespace {

// Launches `kernel` chained to the stream's previous work by programmatic dependent
// launch: it may start while its predecessor finishes, and waits for it (every plan
// kernel calls griddepcontrol.wait before reading anything the predecessor wrote).
template <typename... Args>
cudaError_t launch_pdl(void (*kernel)(Args...), int grid, int block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

#ifdef EWG_DEBUG
cudaError_t launch_lookback_probe(uint32_t* words, int tile, int poll_limit, int* out, cudaStream_t stream) {
  lookback_probe_kernel<<<1, 32, 0, stream>>>(words, tile, poll_limit, out);
  return cudaGetLastError();
}
#endif

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream) {
  if (a.n <= kHashMaxN) return launch_pdl(plan_hashed_kernel, kHashParts, kHashThreads, kHashSmem, stream, a);
  const int tiles = a.tiles;
  cudaError_t e = launch_pdl(pack_kernel, tiles, kPackThreads, 0, stream, a);
  const uint32_t* ks = a.keys_a;
  const uint32_t* vs = a.vals_a;
  uint32_t* kd = a.keys_b;
  uint32_t* vd = a.vals_b;
  for (int pass = 0; pass < a.passes && e == cudaSuccess; ++pass) {
    e = launch_pdl(sweep_kernel, tiles, kSweepThreads, 0, stream, a, ks, vs, kd, vd, pass);
    const uint32_t* nk = kd;
    const uint32_t* nv = vd;
    kd = const_cast<uint32_t*>(ks);
    vd = const_cast<uint32_t*>(vs);
    ks = nk;
    vs = nv;
  }
  if (e == cudaSuccess) e = launch_pdl(list_kernel, tiles, kListThreads, kListDynSmem, stream, a, ks, vs);
  return e;
}

}  // namespace ewg
