// Apply kernel: chunk partial sums, ordered long-run folds, add into main_grad.
//
// Counterpart of _partial_sums_kernel and _long_run_sums_kernel (Megatron Core API
// docs, core.fusions.fused_embedding_wgrad, "Functions").  The arithmetic is the
// module docstring's: per chunk of at most NROWS rows, part = ((0 + g_0) + g_1) + ...
// in fp32 and position order; per token, t = ((0 + part_0) + part_1) + ... in chunk
// order; w = round_to_grad_dtype(t); main_grad[id] = round_to_main_grad_dtype(
// main_grad[id] + w) computed in fp32.
//
// One persistent kernel, a bulk-copy pipeline per CTA, over three kinds of work item:
//   long chunk   (chunk of a long run, column tile): part -> fp32 partial row
//   fold         (long run, 512-column group): the run's partial rows in chunk order,
//                round, add into main_grad
//   short chunk  (chunk of a one-chunk run, column tile): part, round, add into main_grad
// Items are handed out long chunks first and folds in the middle, so a fold's partial
// rows are normally complete when it is claimed; a fold still waits (bounded) on its
// run's arrival counter, which each consumer warp bumps after storing its partial
// columns.  Within a CTA a producer warp issues cp.async.bulk copies of the gathered
// grad row segments (one lane per row) and of the main_grad segment, or of a fold batch
// (one contiguous block of partial rows), into a shared-memory ring, completing on a
// per-slot mbarrier; four consumer warps (8 columns per thread) take the slots in order,
// add the rows in order from shared memory and release the slot.  Each item's segments
// are also requested into L2 before the producer waits for ring space, so the bytes an SM
// keeps in flight are not bounded by its rings.
#include <cuda_bf16.h>

#include "ewg.h"
#include "ewg_internal.cuh"
#include "ewg_ptx.cuh"

namespace ewg {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kSpinLimit = 1u << 22;   // bounded mbarrier waits

enum ItemKind { kEnd = -1, kShortChunk = 0, kLongChunk = 1, kCombine = 2 };

// The producer's lookahead: an item is claimed kClaimAhead steps before its table entry
// is staged in shared memory, and staged kStageAhead steps before it is issued, so
// neither the claim (an atomic on a counter all CTAs share) nor the entry's load stalls
// the issue.  Deeper lookahead was measured to lengthen the end of the kernel: a CTA
// holding claimed items finishes late while others have run dry.
constexpr int kClaimAhead = 2;
constexpr int kStageAhead = 1;
constexpr int kStage = kStageAhead + 1;   // staged entries: in flight + the one issued

// Short chunks of at most kWideRows rows, handed out as whole-row units, are copied in
// tiles twice as wide: half as many items to issue and consume for the same bytes.
constexpr int kWideRows = 2;
// Every item fits the ring: a 10-row chunk over the widest tile (with its main_grad
// segment), a wide tile of kWideRows rows, a fold batch.
static_assert(kNrows * kMaxTileColsBf16 * 2 + kMaxTileColsBf16 * 4 <= kRingBytes &&
                  kNrows * kMaxTileColsFp32 * 4 + kMaxTileColsFp32 * 4 <= kRingBytes &&
                  kWideRows * 2 * kMaxTileColsBf16 * 2 + 2 * kMaxTileColsBf16 * 4 <= kRingBytes &&
                  kWideRows * 2 * kMaxTileColsFp32 * 4 + 2 * kMaxTileColsFp32 * 4 <= kRingBytes &&
                  kCombineBatch * kCombineCols * 4 + kCombineCols * 4 <= kRingBytes,
              "every ring item fits the ring");

struct Item {
  int off;        // byte offset of the item in the ring
  int rows;       // grad rows (chunks) or partial rows (combine) in the ring
  int id;         // main_grad row
  int prow;       // long chunk: its partial row (run's first + c); fold: the batch's block
                  // of partial rows, in 128-byte lines
  int col0;       // first column
  int cols;       // columns
  int kind;
  int flags;      // fold: bit 0 first batch, bit 1 last batch, slice width << 2;
                  // long chunk: its index c in the run (and `id` holds the run's C)
};

struct Smem {
  int4 desc[kStage][kChunkWords / 4];   // staged chunk descriptors / long-run rows
  int kind[kStage];                     // the staged items' kinds ...
  int tile[kStage];                     // ... and column tiles (fold: column group)
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
  Item info[kSlots];
  int prefix[3][kMaxParts + 1];   // long chunks, short chunks, long runs
  int offset[3][kMaxParts];
  int num_parts;
  int abort;
  int epoch;      // apply calls already made on this plan
  int spin_limit; // polls of a fold's arrival counter before it gives up
};

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

// Waits for the phase of `bar` with the given parity; false if the wait gave up
// (limit reached or another thread of the CTA aborted).
__device__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort) return false;
  }
  return false;
}

__device__ void give_up(const ApplyArgs& a, volatile int* abort) {
  *abort = 1;
  atomicExch(const_cast<int*>(&a.header->status), kStatusTimeout);
}

// Adds 8 elements of a row held in shared memory, in order, into acc.
template <bool BF16>
__device__ __forceinline__ void add_row(float acc[8], const unsigned char* p) {
  if constexpr (BF16) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    acc[0] = acc[0] + bf16_lo(v.x);
    acc[1] = acc[1] + bf16_hi(v.x);
    acc[2] = acc[2] + bf16_lo(v.y);
    acc[3] = acc[3] + bf16_hi(v.y);
    acc[4] = acc[4] + bf16_lo(v.z);
    acc[5] = acc[5] + bf16_hi(v.z);
    acc[6] = acc[6] + bf16_lo(v.w);
    acc[7] = acc[7] + bf16_hi(v.w);
  } else {
    const float4 x = *reinterpret_cast<const float4*>(p);
    const float4 y = *reinterpret_cast<const float4*>(p + 16);
    acc[0] = acc[0] + x.x;
    acc[1] = acc[1] + x.y;
    acc[2] = acc[2] + x.z;
    acc[3] = acc[3] + x.w;
    acc[4] = acc[4] + y.x;
    acc[5] = acc[5] + y.y;
    acc[6] = acc[6] + y.z;
    acc[7] = acc[7] + y.w;
  }
}

// w = round_g(t); out = round_mg(m + w) in fp32, m from the ring; stored to main_grad.
template <bool GBF16, bool MBF16>
__device__ __forceinline__ void finish(const ApplyArgs& a, const float t[8],
                                       const unsigned char* m_smem, int id, int col) {
  float w[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) w[e] = GBF16 ? __bfloat162float(__float2bfloat16_rn(t[e])) : t[e];
  if constexpr (MBF16) {
    const uint4 m = *reinterpret_cast<const uint4*>(m_smem);
    uint4 o;
    o.x = pack_bf16(bf16_lo(m.x) + w[0], bf16_hi(m.x) + w[1]);
    o.y = pack_bf16(bf16_lo(m.y) + w[2], bf16_hi(m.y) + w[3]);
    o.z = pack_bf16(bf16_lo(m.z) + w[4], bf16_hi(m.z) + w[5]);
    o.w = pack_bf16(bf16_lo(m.w) + w[6], bf16_hi(m.w) + w[7]);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.main_grad) +
                              static_cast<long long>(id) * a.mg_stride + col) = o;
  } else {
    float4 m0 = *reinterpret_cast<const float4*>(m_smem);
    float4 m1 = *reinterpret_cast<const float4*>(m_smem + 16);
    m0.x = m0.x + w[0];
    m0.y = m0.y + w[1];
    m0.z = m0.z + w[2];
    m0.w = m0.w + w[3];
    m1.x = m1.x + w[4];
    m1.y = m1.y + w[5];
    m1.z = m1.z + w[6];
    m1.w = m1.w + w[7];
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.main_grad) +
                                            static_cast<long long>(id) * a.mg_stride + col);
    dst[0] = m0;
    dst[1] = m1;
  }
}

// Index of list element `ord` (< the list's length) given the per-partition prefix
// counts and offsets, found by the whole warp: the partition holding `ord` is the last
// one whose prefix is at most `ord` (an empty partition shares its prefix with the
// next, so it is never the last such one unless it is the last partition, which then
// holds `ord`).
__device__ __forceinline__ int list_index(const int* prefix, const int* offset, int parts, int ord,
                                          int lane) {
  int n = 0;
  for (int p0 = 0; p0 < parts; p0 += 32) {
    const int p = p0 + lane;
    n += __popc(__ballot_sync(kFull, p < parts && prefix[p] <= ord));
  }
  return offset[n - 1] + (ord - prefix[n - 1]);
}

// The producer warp of a CTA.  Its 32 lanes take the same steps in lockstep, so every
// lane holds the same ring bookkeeping; lane 0 publishes item info and arms the slot
// barriers, and the lanes issue the bulk copies of an item's rows side by side (lane k
// copies row k), which keeps the serial instruction path per item short.
template <bool GBF16, bool MBF16>
struct Producer {
  const ApplyArgs& a;
  Smem& s;
  unsigned char* ring;
  const int lane;
  int q = 0;            // items issued
  int rel = 0;          // items known to be consumed
  uint32_t head = 0, tail = 0;
  uint64_t pol;
  bool ok = true;

  __device__ Producer(const ApplyArgs& args, Smem& sm, unsigned char* r)
      : a(args), s(sm), ring(r), lane(static_cast<int>(threadIdx.x & 31)),
        pol(ptx::policy_evict_first()) {}

  // Lane 0 waits (bounded) for the oldest item in the ring to be consumed.
  __device__ bool confirm_oldest() {
    const int slot = rel % kSlots;
    int got = 0;
    if (lane == 0) got = wait_phase(&s.empty[slot], (rel / kSlots) & 1, &s.abort);
    if (!__shfl_sync(kFull, got, 0)) return false;
    ++rel;
    head = rel < q ? static_cast<uint32_t>(s.info[rel % kSlots].off) : tail;
    return true;
  }

  // Offset of `bytes` free, contiguous ring bytes (items leave in issue order).
  __device__ int reserve(uint32_t bytes) {
    while (q - rel >= kSlots)
      if (!confirm_oldest()) return -1;
    for (;;) {
      if (q == rel) head = tail = 0;
      const bool full = q > rel && head == tail;
      if (!full) {
        if (head <= tail) {
          if (tail + bytes <= static_cast<uint32_t>(kRingBytes)) return static_cast<int>(tail);
          if (bytes <= head) return 0;
        } else if (tail + bytes <= head) {
          return static_cast<int>(tail);
        }
      }
      if (!confirm_oldest()) return -1;
    }
  }

  // Publishes the item and arms its slot's barrier for `bytes`; the copies follow.
  __device__ uint64_t* open(const Item& it, uint32_t bytes) {
    const int slot = q % kSlots;
    // The consumers' reads of this ring space are ordered before the new copies by the
    // slot's empty barrier, which lane 0 has waited on.
    if (lane == 0) {
      s.info[slot] = it;
      ptx::mbar_arrive_expect_tx(&s.full[slot], bytes);
    }
    __syncwarp();
    tail = static_cast<uint32_t>(it.off) + bytes;
    ++q;
    return &s.full[slot];
  }

  // One (chunk, column tile) item: the chunk's grad row segments (lane k: row k), plus
  // the main_grad segment (lane len) when the run has no other chunk.
  __device__ bool chunk_item(const int* d, int tile, int tc, bool is_long) {
    const int col0 = tile * tc;
    const int cols = min(tc, a.hidden - col0);
    const int meta = d[kDescMeta];
    int len = meta & 15;
    int id = d[kDescId];
    int prow = d[kDescPartial], C = d[kDescNumChunks], ci = meta >> 4;
    if (!checked(len >= 1 && len <= kNrows, a.header)) len = 1;
    if (!checked(is_long || (id >= 0 && id < a.num_embeddings), a.header)) id = 0;
    if (!checked(!is_long || (C >= 1 && ci < C && prow - ci >= 0 && prow - ci + C <= a.partial_cap), a.header))
      prow = ci = 0, C = 1;
    const uint32_t row_bytes = cols * (GBF16 ? 2 : 4);
    const uint32_t mg_bytes = is_long ? 0u : cols * (MBF16 ? 2 : 4);
    const uint32_t bytes = len * row_bytes + mg_bytes;
    const char* src = nullptr;   // this lane's segment: grad row `lane`, or the main_grad row
    if (lane < len) {
      long long p = d[kDescPos + lane];
      if (!checked(p >= 0 && p < a.n, a.header)) p = 0;
      src = static_cast<const char*>(a.grad) + (p * a.grad_stride + col0) * (GBF16 ? 2 : 4);
    } else if (lane == len && !is_long) {
      src = static_cast<const char*>(a.main_grad) +
            (static_cast<long long>(id) * a.mg_stride + col0) * (MBF16 ? 2 : 4);
    }
    const uint32_t src_bytes = lane < len ? row_bytes : mg_bytes;
    // The segments start towards L2 before the wait for ring space: the bytes a CTA has
    // in flight are then not limited by its ring, and the copies below mostly hit L2.
    if (src) ptx::bulk_prefetch_l2(src, src_bytes, pol);
    const int off = reserve(bytes);
    if (off < 0) return false;
    // for a long chunk, flags holds its index c in the run (prow - c: the run's counter)
    Item it{off, len, is_long ? C : id, prow, col0, cols, is_long ? kLongChunk : kShortChunk,
            is_long ? ci : 0};
    uint64_t* bar = open(it, bytes);
    if (src) ptx::bulk_g2s(ring + off + lane * row_bytes, src, src_bytes, bar, pol);
    return true;
  }

  // Waits until every consumer warp that handled a chunk item of the run has stored its
  // partial columns: C chunks x Tl column tiles x kConsumerWarps arrivals.  Lane 0 polls
  // with acquire loads (at most spin_limit times, and it stops early once this CTA or any
  // other has given up), then orders its later bulk copies of the partial rows (async
  // proxy) after the rows' generic-proxy stores.  Lane 0 alone copies partial rows; the
  // other copy of a fold, the main_grad segment, reads nothing the run's chunks write.
  __device__ bool wait_run(int prow0, int target) {
    const int* cnt = a.arrivals + prow0;
    const volatile int* status = &a.header->status;
    int got = 0;
    if (lane == 0) {
      for (int i = 0; i < s.spin_limit; ++i) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
        if (v >= target) {
          got = 1;
          break;
        }
        if ((i & 63) == 63 && (s.abort || *status == kStatusTimeout)) break;
        __nanosleep(64);
      }
      if (got) asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    return __shfl_sync(kFull, got, 0) != 0;
  }

  // One fold: a column slice (the whole 512-column group, or the entry's 1/split of it)
  // of a long run, as batches of consecutive partial rows, each one bulk copy of a
  // contiguous block (partial rows are slice-major); the last batch also brings the
  // main_grad segment.
  __device__ bool combine_task(const int* run, int group, int Tl) {
    const int prow0 = run[0], C = run[1], id = run[2];
    const int split = run[3] >> 4, width = kCombineCols / split;
    if (!checked(prow0 >= 0 && C >= 1 && prow0 + C <= a.partial_cap && id >= 0 && id < a.num_embeddings &&
                     (split == 1 || split == 2 || split == 4) && (run[3] & 15) < split,
                 a.header))
      return true;   // nothing is issued for a fold whose table entry is out of range
    const int col0 = group * kCombineCols + (run[3] & 15) * width;
    const int cols = min(width, a.hidden - col0);
    if (cols <= 0) return true;   // a slice past the last column: nothing to fold
    if (!wait_run(prow0, (s.epoch + 1) * C * Tl * kConsumerWarps)) {
      if (lane == 0) give_up(a, &s.abort);
      return false;
    }
    const uint32_t row_bytes = width * 4;   // the slice's partial rows are `width` apart
    const uint32_t mg_bytes = cols * (MBF16 ? 2 : 4);
    const int batch = min(kCombineBatch * split, 31);   // about 16 KB of partial rows
    // the slice's block: C rows of `width` floats (a multiple of 32: whole 128-byte lines)
    const long long block = static_cast<long long>(prow0) * partial_row_floats(a.hidden) +
                            static_cast<long long>(C) * col0;
    for (int b0 = 0; b0 < C; b0 += batch) {
      const int nb = min(batch, C - b0);
      const bool last = b0 + nb == C;
      const uint32_t bytes = nb * row_bytes + (last ? mg_bytes : 0u);
      const int off = reserve(bytes);
      if (off < 0) return false;
      const long long at = block + static_cast<long long>(b0) * width;
      Item it{off, nb, id, static_cast<int>(at / 32), col0, cols, kCombine,
              (b0 == 0 ? 1 : 0) | (last ? 2 : 0) | (width << 2)};
      uint64_t* bar = open(it, bytes);
      if (lane == 0) {
        ptx::bulk_g2s(ring + off, a.partial + at, nb * row_bytes, bar, pol);
      } else if (lane == 1 && last) {
        const char* m = static_cast<const char*>(a.main_grad);
        ptx::bulk_g2s(ring + off + nb * row_bytes,
                      m + (static_cast<long long>(id) * a.mg_stride + col0) * (MBF16 ? 2 : 4),
                      mg_bytes, bar, pol);
      }
    }
    return true;
  }

  __device__ void finish_stream() {
    if (ok) {
      while (q - rel >= kSlots)
        if (!confirm_oldest()) {
          ok = false;
          break;
        }
    }
    if (ok) {
      if (lane == 0) {
        const int slot = q % kSlots;
        s.info[slot].kind = kEnd;
        ptx::mbar_arrive(&s.full[slot]);
      }
      ++q;
      return;
    }
    // gave up: let the copies already in flight land before the CTA exits
    if (lane == 0) {
      for (int r = rel; r < q; ++r) {
        uint64_t* bar = &s.full[r % kSlots];
        for (uint32_t i = 0; i < kSpinLimit && !ptx::mbar_try_wait(bar, (r / kSlots) & 1); ++i) {
        }
      }
    }
  }
};

template <bool GBF16, bool MBF16>
__device__ void produce(const ApplyArgs& a, Smem& s, unsigned char* ring, int first_claim) {
  Producer<GBF16, MBF16> P(a, s, ring);
  const int lane = P.lane;
  const int parts = s.num_parts;
  const int Tl = (a.hidden + a.tile_cols_long - 1) / a.tile_cols_long;
  const int Ts = (a.hidden + a.tile_cols_rest - 1) / a.tile_cols_rest;
  const int Tc = (a.hidden + kCombineCols - 1) / kCombineCols;
  // wide tiles: half as many as Ts, for units of at most kWideRows rows
  const int Tw = (Ts + 1) / 2;
  const int tcw = ((a.hidden + Tw - 1) / Tw + 7) / 8 * 8;
  // Work items, in the order they are handed out (counts fit in 32 bits, checked on the
  // host).  A "unit" is one short-run chunk over all its column tiles (one claim, one
  // descriptor, Ts tile copies); a "tile item" is one chunk over one column tile; a
  // fold is one (long run, 512-column group).  The first G0 = min(G, short chunks)
  // items are the static first items of CTAs 0..G0-1; every other item is claimed from
  // the kernel's counter, so a CTA owns a long-run chunk only once it is running.  A
  // fold waits only for chunks handed out before it, each owned by a running CTA that
  // processes its items in claim order and never waits on a chunk item: the waits end
  // whether or not all CTAs are resident.  The last short chunks go out as tile items,
  // so the work ends in small pieces.
  //   [0, G0)                units: short chunks 0..G0-1 (static)
  //   [G0, G0+L)             tile items of the long runs' chunks -> partial rows
  //   [G0+L, G0+L+S1)        units: short chunks G0..G0+S1-1
  //   [G0+L+S1, G0+L+S1+F)   folds of the long runs (their partial rows are mostly done
  //                          by then; a fold waits for the rest on the run's counter)
  //   [G0+L+S1+F, total)     tile items of the remaining short chunks
  const int L = s.prefix[0][parts] * Tl;
  const int S = s.prefix[1][parts];   // short chunks
  const int F = s.prefix[2][parts] * Tc;
  const int G = static_cast<int>(gridDim.x);
  const int G0 = min(G, S);
  const int S1 = (S - G0) / 2;
  const int R0 = G0 + L + S1 + F;     // first tile item of the remaining short chunks
  const int total = R0 + (S - G0 - S1) * Ts;
  int* work = const_cast<int*>(&a.header->work[0]);

  // Stages the table entry of `item` (its chunk descriptor, or its long-run row) in
  // shared-memory stage `st` with asynchronous copies (one commit group per lane and
  // call), and records the item's kind and column tile (fold: column group; unit: -1).
  auto stage = [&](int item, int st) {
    __syncwarp();   // every lane's reads of this stage's previous entry are done
    int kind = kEnd, tile = -1;
    if (item < total) {
      int list, e;
      if (item < G0) {
        kind = kShortChunk, list = 1, e = item;
      } else if (item < G0 + L) {
        kind = kLongChunk, list = 0, e = (item - G0) / Tl;
        tile = item - G0 - e * Tl;
      } else if (item < G0 + L + S1) {
        kind = kShortChunk, list = 1, e = item - L;
      } else if (item < R0) {
        kind = kCombine, list = 2, e = (item - G0 - L - S1) / Tc;
        tile = item - G0 - L - S1 - e * Tc;
      } else {
        const int o = item - R0, q = o / Ts;
        kind = kShortChunk, list = 1, e = G0 + S1 + q;
        tile = o - q * Ts;
      }
      const int idx = list_index(s.prefix[list], s.offset[list], parts, e, lane);
      if (kind == kCombine) {
        if (lane == 0) ptx::cp_async16(&s.desc[st][0], reinterpret_cast<const int4*>(a.runs) + idx, P.pol);
      } else if (lane < kChunkWords / 4) {
        const int4* src = reinterpret_cast<const int4*>(a.chunks + static_cast<long long>(idx) * kChunkWords);
        ptx::cp_async16(&s.desc[st][lane], src + lane, P.pol);
      }
    }
    if (lane == 0) {
      s.kind[st] = kind;
      s.tile[st] = tile;
    }
    ptx::cp_async_commit();
  };
  // Issues the item staged in `st`: 1 issued, 0 end of the work, -1 gave up.
  auto issue = [&](int st, bool newest) {
    // this lane's copies for `st`: the newest group (nothing staged since), or the one
    // staged kStageAhead steps ago
    if (newest) ptx::cp_async_wait<0>();
    else ptx::cp_async_wait<kStageAhead>();
    __syncwarp();                        // ... and every other lane's
    const int kind = s.kind[st], tile = s.tile[st];
    if (kind == kEnd) return 0;
    const int* d = reinterpret_cast<const int*>(&s.desc[st][0]);
    bool ok = true;
    if (kind == kCombine) {
      ok = P.combine_task(d, tile, Tl);
    } else if (tile >= 0) {
      ok = P.chunk_item(d, tile, kind == kLongChunk ? a.tile_cols_long : a.tile_cols_rest,
                        kind == kLongChunk);
    } else {   // a unit: every column tile of the short chunk; few rows take wide tiles
      const bool wide = (d[kDescMeta] & 15) <= kWideRows;
      const int tc = wide ? tcw : a.tile_cols_rest, T = wide ? Tw : Ts;
      for (int tt = 0; tt < T && ok; ++tt) ok = P.chunk_item(d, tt, tc, false);
    }
    return ok ? 1 : -1;
  };

  // Step k stages the item claimed kClaimAhead steps earlier (lane 0 holds it in
  // c[k % kClaimAhead]), claims the item it will stage kClaimAhead steps later into the
  // same register, and issues the item staged kStageAhead steps earlier.  The loop over
  // c is unrolled so each claim keeps its own register and is read only when it is due.
  // Claims increase within a CTA; once one is past the end, so are the later ones.
  int c[kClaimAhead];
#pragma unroll
  for (int j = 0; j < kClaimAhead; ++j) c[j] = total;
  if (lane == 0) {   // first_claim: this CTA's first counter claim, made in the prologue
    const bool fixed = static_cast<int>(blockIdx.x) < G0;
    c[0] = fixed ? static_cast<int>(blockIdx.x) : G0 + first_claim;
    c[1] = fixed ? G0 + first_claim : G0 + atomicAdd(work, 1);
#pragma unroll
    for (int j = 2; j < kClaimAhead; ++j) c[j] = G0 + atomicAdd(work, 1);
  }
  int k = 0;
  bool more = true;
  while (more) {
#pragma unroll
    for (int j = 0; j < kClaimAhead; ++j) {
      if (more) {
        if (k == kStageAhead) {   // the first item goes out before the next claim is read
          const int r = issue(0, true);
          if (r <= 0) {
            more = false;
            P.ok = r == 0;
            continue;
          }
        }
        const int v = __shfl_sync(kFull, c[j], 0);
        stage(v, k % kStage);
        if (lane == 0) c[j] = v < total ? G0 + atomicAdd(work, 1) : total;
        if (k > kStageAhead) {
          const int r = issue((k - kStageAhead) % kStage, false);
          if (r <= 0) {
            more = false;
            P.ok = r == 0;
          }
        }
        ++k;
      }
    }
  }
  ptx::cp_async_wait<0>();
  P.finish_stream();
}

template <bool GBF16, bool MBF16>
__device__ void consume(const ApplyArgs& a, Smem& s, const unsigned char* ring) {
  const int t = threadIdx.x, lane = t & 31;
  const uint64_t pol_keep = ptx::policy_evict_last();
  float total[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) total[e] = 0.0f;
  for (int q = 0;; ++q) {
    const int slot = q % kSlots;
    if (!wait_phase(&s.full[slot], (q / kSlots) & 1, &s.abort)) {
      give_up(a, &s.abort);
      return;
    }
    const Item it = s.info[slot];
    if (it.kind == kEnd) return;
    const unsigned char* base = ring + it.off;
    if (it.kind == kCombine) {   // at most kCombineCols <= 8 * kConsumers columns
      const int c = t * 8;
      const uint32_t row_bytes = (it.flags >> 2) * 4;   // slice width apart
      if (c < it.cols) {
        if (it.flags & 1) {
#pragma unroll
          for (int e = 0; e < 8; ++e) total[e] = 0.0f;   // the combine starts from 0
        }
        for (int k = 0; k < it.rows; ++k) add_row<false>(total, base + k * row_bytes + c * 4);
        if (it.flags & 2)
          finish<GBF16, MBF16>(a, total, base + it.rows * row_bytes + c * (MBF16 ? 2 : 4), it.id,
                               it.col0 + c);
      }
      // The batch's partial rows are dead now: drop their L2 lines (the block is whole
      // 128-byte lines) instead of writing them back.
      {
        const float* blk = a.partial + static_cast<long long>(it.prow) * 32;
        const int lines = it.rows * static_cast<int>(row_bytes) / 128;
        for (int l = t; l < lines; l += kConsumers) ptx::discard_l2_line(blk + l * 32);
      }
    } else {   // chunk item: passes of 8 * kConsumers columns over the tile
      const uint32_t row_bytes = it.cols * (GBF16 ? 2 : 4);
      for (int c = t * 8; c < it.cols; c += 8 * kConsumers) {
        float part[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) part[e] = 0.0f;
        for (int k = 0; k < it.rows; ++k)
          add_row<GBF16>(part, base + k * row_bytes + c * (GBF16 ? 2 : 4));
        if (it.kind == kLongChunk) {
          // partial rows are read back soon by the run's fold: ask L2 to keep them.  Slice-
          // major: chunk c's slice [s, s + w) at C s + c w in the run's floats.
          const int C = it.id, ci = it.flags, w = kCombineCols / fold_entries(C);
          const int col = it.col0 + c, s0 = col & ~(w - 1);
          float* dst = a.partial + static_cast<long long>(it.prow - ci) * partial_row_floats(a.hidden) +
                       static_cast<long long>(C) * s0 + static_cast<long long>(ci) * w + (col - s0);
          ptx::st_global_v4(dst, part[0], part[1], part[2], part[3], pol_keep);
          ptx::st_global_v4(dst + 4, part[4], part[5], part[6], part[7], pol_keep);
        } else {   // the run's only chunk: t = 0 + part
          float tt[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) tt[e] = 0.0f + part[e];
          finish<GBF16, MBF16>(a, tt, base + it.rows * row_bytes + c * (MBF16 ? 2 : 4), it.id,
                               it.col0 + c);
        }
      }
      if (it.kind == kLongChunk) {   // publish this warp's partial columns to the fold
        // every lane's stores precede lane 0's release add (the warp barrier orders them
        // first); the fold's acquire load of the counter pairs with it
        __syncwarp();
        if (lane == 0) ptx::red_release_add(a.arrivals + (it.prow - it.flags), 1);
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&s.empty[slot]);
  }
}

template <bool GBF16, bool MBF16>
__global__ void __launch_bounds__(kApplyThreads, kApplyCtasPerSm) apply_kernel(ApplyArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* ring = smem_raw;
  Smem& s = *reinterpret_cast<Smem*>(smem_raw + kRingBytes);
  const int t = threadIdx.x;
  if (t == 0) {
    for (int i = 0; i < kSlots; ++i) {
      ptx::mbar_init(&s.full[i], 1);
      ptx::mbar_init(&s.empty[i], kConsumerWarps);
    }
    ptx::fence_mbar_init();
    s.abort = 0;
  }
  // Launched early on the SMs the plan leaves free; the plan's lists are read only
  // after it has completed.  Meanwhile the producer warp pulls this CTA's share of the
  // first prefetch_rows grad rows into L2 (one bulk prefetch per row and lane).
  if (t >= kConsumers && a.prefetch_rows > 0) {
    const long long rows = a.prefetch_rows, G = gridDim.x;
    const int r1 = static_cast<int>(rows * (blockIdx.x + 1) / G);
    const uint32_t row_bytes = static_cast<uint32_t>(a.hidden) * (GBF16 ? 2u : 4u);
    const uint64_t keep = ptx::policy_evict_last();
    const char* g = static_cast<const char*>(a.grad);
    for (int r = static_cast<int>(rows * blockIdx.x / G) + (t - kConsumers); r < r1; r += 32)
      ptx::bulk_prefetch_l2(g + static_cast<long long>(r) * a.grad_stride * (GBF16 ? 2 : 4), row_bytes,
                            keep);
  }
  ptx::pdl_wait_prior_grid();

  // The header check, the partition tables and the producer's first dynamic claim all
  // go out at once: one round trip to L2 instead of one per dependent load.
  const Header* h = a.header;
  int first_claim = 0;
  if (t == kConsumers) first_claim = atomicAdd(const_cast<int*>(&h->work[0]), 1);
  if (t == 0) {   // one reader decides for the whole CTA
    const int status = h->status, hn = h->n, hh = h->hidden, np = h->num_parts, ep = h->epoch,
              sl = h->spin_limit;
    const long long hv = h->num_embeddings;
    int go = status == EWG_OK;
    if (go && (hn != a.n || hh != a.hidden || hv != a.num_embeddings || np != a.parts)) {
      if (blockIdx.x == 0) const_cast<Header*>(h)->status = kStatusInvalid;
      go = 0;
    }
    s.num_parts = go ? np : -1;
    s.epoch = ep;
    s.spin_limit = sl;
  }
  {   // counts (into prefix, scanned below) and offsets of the three lists, for the
      // partitions the plan of this size writes (every CTA reads these same lines)
    constexpr int kPer = (3 * kHashParts + kApplyThreads - 1) / kApplyThreads;
    static_assert(kHashParts <= kMaxParts, "partition tables");
    const int parts = a.parts, entries = 3 * parts;
    int cnt[kPer], off[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int i = t + r * kApplyThreads;
      const int list = i / parts, p = i - list * parts;
      const int ct = list == 0 ? kLongCnt : list == 1 ? kShortCnt : kRunCnt;
      const int ot = list == 0 ? kLongOff : list == 1 ? kShortOff : kRunOff;
      cnt[r] = i < entries ? a.tables[ct * kMaxParts + p] : 0;
      off[r] = i < entries ? a.tables[ot * kMaxParts + p] : 0;
    }
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int i = t + r * kApplyThreads;
      if (i < entries) {
        const int list = i / parts, p = i - list * parts;
        s.prefix[list][p] = cnt[r];
        s.offset[list][p] = off[r];
      }
    }
  }
  __syncthreads();
  if (s.num_parts < 0) return;
  if (t < 3 * 32) {   // warp `list`: counts -> exclusive prefix, in place
    const int list = t >> 5, lane = t & 31, parts = s.num_parts;
    int carry = 0;
    for (int p0 = 0; p0 < parts; p0 += 32) {
      const int p = p0 + lane;
      const int c = p < parts ? s.prefix[list][p] : 0;
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
      }
      if (p < parts) s.prefix[list][p] = carry + x - c;
      carry += __shfl_sync(kFull, x, 31);
    }
    if (lane == 0) s.prefix[list][parts] = carry;
  }
  __syncthreads();

  if (t >= kConsumers) {
    produce<GBF16, MBF16>(a, s, ring, first_claim);   // the whole producer warp
    return;
  }
  consume<GBF16, MBF16>(a, s, ring);
  // The last CTA to finish re-arms the work counter and the long runs' arrival counters,
  // so that one plan can serve further ewg_apply calls.  Every CTA claims its last item
  // before its consumers see the end of its stream, so no claim can follow this reset.
  if (t == 0) {
    Header* hw = const_cast<Header*>(h);
    if (atomicAdd(&hw->done, 1) == static_cast<int>(gridDim.x) - 1) {
      hw->work[0] = 0;
      hw->done = 0;
      hw->epoch = s.epoch + 1;   // the arrival counters of the next call start here
    }
  }
}

constexpr size_t kApplySmem = kRingBytes + sizeof(Smem);

template <bool G, bool M>
cudaError_t launch_one(const ApplyArgs& a, int num_sms, cudaStream_t stream) {
  static int blocks_per_sm = 0;
  if (blocks_per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(apply_kernel<G, M>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kApplySmem));
    if (e != cudaSuccess) return e;
    int b = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, apply_kernel<G, M>, kApplyThreads,
                                                      kApplySmem);
    if (e != cudaSuccess) return e;
    blocks_per_sm = b > 0 ? b : 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms * blocks_per_sm);
  cfg.blockDim = dim3(kApplyThreads);
  cfg.dynamicSmemBytes = kApplySmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, apply_kernel<G, M>, a);
}

}  // namespace

cudaError_t launch_apply(const ApplyArgs& a, int grad_bf16, int mg_bf16, int num_sms,
                         cudaStream_t stream) {
  if (grad_bf16) {
    return mg_bf16 ? launch_one<true, true>(a, num_sms, stream)
                   : launch_one<true, false>(a, num_sms, stream);
  }
  return mg_bf16 ? launch_one<false, true>(a, num_sms, stream)
                 : launch_one<false, false>(a, num_sms, stream);
}

}  // namespace ewg
