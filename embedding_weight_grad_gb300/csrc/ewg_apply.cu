// Apply kernel: chunk partial sums, ordered long-run combine, add into main_grad.
//
// Counterpart of _partial_sums_kernel and _long_run_sums_kernel (Megatron Core API
// docs, core.fusions.fused_embedding_wgrad, "Functions"), fused into one persistent
// kernel.  The arithmetic is the module docstring's: per chunk of at most NROWS rows,
// part = ((0 + g_0) + g_1) + ... in fp32 and position order; per token,
// t = ((0 + part_0) + part_1) + ... in chunk order; w = round_to_grad_dtype(t);
// main_grad[id] = round_to_main_grad_dtype(main_grad[id] + w) in fp32.
//
// Work item = (chunk, 256-column slice), one warp each; lane l owns 8 consecutive
// columns, so every gathered grad row is read as one 16-byte load per lane (bf16)
// and a warp covers 512 contiguous bytes of it.  All rows of a chunk are loaded
// before the first add.  A token with a single chunk is finished by the warp that
// summed it.  For a longer token each warp stores its fp32 partial row, and the
// last warp to arrive at the (token, slice) counter adds all of the token's
// partials in chunk order; which warp that is does not change any value.
#include <cuda_bf16.h>

#include "ewg.h"
#include "ewg_internal.cuh"

namespace ewg {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

__device__ __forceinline__ uint4 load_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// fp32 partial sum of one chunk's rows over this lane's 8 columns.  `word` holds
// descriptor word `lane`; words 0..9 are the chunk's token positions.
template <bool GBF16>
__device__ __forceinline__ void chunk_partial(const ApplyArgs& a, int word, int len, int col,
                                              bool active, float part[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) part[e] = 0.0f;
  if constexpr (GBF16) {
    const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(a.grad) + col;
    uint4 v[kNrows];
#pragma unroll
    for (int k = 0; k < kNrows; ++k) {
      const int p = __shfl_sync(kFull, word, kDescPos + k);
      v[k] = make_uint4(0, 0, 0, 0);
      if (k < len && active) v[k] = load_stream_u4(g + static_cast<long long>(p) * a.grad_stride);
    }
#pragma unroll
    for (int k = 0; k < kNrows; ++k) {
      if (k < len) {
        part[0] = part[0] + bf16_lo(v[k].x);
        part[1] = part[1] + bf16_hi(v[k].x);
        part[2] = part[2] + bf16_lo(v[k].y);
        part[3] = part[3] + bf16_hi(v[k].y);
        part[4] = part[4] + bf16_lo(v[k].z);
        part[5] = part[5] + bf16_hi(v[k].z);
        part[6] = part[6] + bf16_lo(v[k].w);
        part[7] = part[7] + bf16_hi(v[k].w);
      }
    }
  } else {
    const float* g = static_cast<const float*>(a.grad) + col;
    uint4 v[kNrows][2];
#pragma unroll
    for (int k = 0; k < kNrows; ++k) {
      const int p = __shfl_sync(kFull, word, kDescPos + k);
      v[k][0] = v[k][1] = make_uint4(0, 0, 0, 0);
      if (k < len && active) {
        const float* r = g + static_cast<long long>(p) * a.grad_stride;
        v[k][0] = load_stream_u4(r);
        v[k][1] = load_stream_u4(r + 4);
      }
    }
#pragma unroll
    for (int k = 0; k < kNrows; ++k) {
      if (k < len) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          part[4 * h + 0] = part[4 * h + 0] + __uint_as_float(v[k][h].x);
          part[4 * h + 1] = part[4 * h + 1] + __uint_as_float(v[k][h].y);
          part[4 * h + 2] = part[4 * h + 2] + __uint_as_float(v[k][h].z);
          part[4 * h + 3] = part[4 * h + 3] + __uint_as_float(v[k][h].w);
        }
      }
    }
  }
}

// w = round_g(t); main_grad[id][col..col+8) = round_mg(main_grad + w) in fp32.
template <bool GBF16, bool MBF16>
__device__ __forceinline__ void finish(const ApplyArgs& a, int id, int col, const float t[8]) {
  float w[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    w[e] = GBF16 ? __bfloat162float(__float2bfloat16_rn(t[e])) : t[e];
  }
  if constexpr (MBF16) {
    uint4* p = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.main_grad) +
                                        static_cast<long long>(id) * a.mg_stride + col);
    const uint4 m = *p;
    uint4 o;
    o.x = pack_bf16(bf16_lo(m.x) + w[0], bf16_hi(m.x) + w[1]);
    o.y = pack_bf16(bf16_lo(m.y) + w[2], bf16_hi(m.y) + w[3]);
    o.z = pack_bf16(bf16_lo(m.z) + w[4], bf16_hi(m.z) + w[5]);
    o.w = pack_bf16(bf16_lo(m.w) + w[6], bf16_hi(m.w) + w[7]);
    *p = o;
  } else {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(a.main_grad) +
                                          static_cast<long long>(id) * a.mg_stride + col);
    float4 m0 = p[0], m1 = p[1];
    m0.x = m0.x + w[0];
    m0.y = m0.y + w[1];
    m0.z = m0.z + w[2];
    m0.w = m0.w + w[3];
    m1.x = m1.x + w[4];
    m1.y = m1.y + w[5];
    m1.z = m1.z + w[6];
    m1.w = m1.w + w[7];
    p[0] = m0;
    p[1] = m1;
  }
}

template <bool GBF16, bool MBF16>
__global__ void __launch_bounds__(kApplyThreads) apply_kernel(ApplyArgs a) {
  Header* hdr = const_cast<Header*>(a.header);
  if (hdr->status != EWG_OK) return;
  if (hdr->n != a.n || hdr->hidden != a.hidden || hdr->num_embeddings != a.num_embeddings) {
    if (blockIdx.x == 0 && threadIdx.x == 0) hdr->status = EWG_ERR_INVALID;
    return;
  }
  const int S = a.slices;
  const long long items = static_cast<long long>(hdr->num_chunks) * S;
  const int lane = threadIdx.x & 31;
  constexpr int kWarps = kApplyThreads / 32;
  const long long first = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const long long stride = static_cast<long long>(gridDim.x) * kWarps;

  for (long long it = first; it < items; it += stride) {
    const int ci = static_cast<int>(it / S);
    const int j = static_cast<int>(it - static_cast<long long>(ci) * S);
    const int word = lane < kChunkWords ? a.chunks[static_cast<long long>(ci) * kChunkWords + lane] : 0;
    const int id = __shfl_sync(kFull, word, kDescId);
    const int meta = __shfl_sync(kFull, word, kDescMeta);
    const int lc = __shfl_sync(kFull, word, kDescLong);
    const int C = __shfl_sync(kFull, word, kDescNumChunks);
    const int len = meta & 15, c = meta >> 4;
    const int col = j * kSliceCols + lane * 8;
    const bool active = col < a.hidden;

    float part[8];
    chunk_partial<GBF16>(a, word, len, col, active, part);

    if (lc < 0) {  // the token's only chunk: t = 0 + part
      float t[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) t[e] = 0.0f + part[e];
      if (active) finish<GBF16, MBF16>(a, id, col, t);
      continue;
    }

    const long long lc0 = lc - c;  // partial row of the token's first chunk
    if (active) {
      float4* dst = reinterpret_cast<float4*>(a.partial + static_cast<long long>(lc) * a.hidden + col);
      dst[0] = make_float4(part[0], part[1], part[2], part[3]);
      dst[1] = make_float4(part[4], part[5], part[6], part[7]);
    }
    __threadfence();
    __syncwarp();
    int prior = 0;
    if (lane == 0) prior = atomicAdd(a.counters + lc0 * S + j, 1);
    prior = __shfl_sync(kFull, prior, 0);
    if (prior != C - 1) continue;  // another warp will arrive later and combine

    __threadfence();
    if (active) {
      const float* src = a.partial + lc0 * a.hidden + col;
      float t[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) t[e] = 0.0f;
#pragma unroll 4
      for (int q = 0; q < C; ++q) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(src + static_cast<long long>(q) * a.hidden));
        const float4 y = __ldcg(reinterpret_cast<const float4*>(src + static_cast<long long>(q) * a.hidden + 4));
        t[0] = t[0] + x.x;
        t[1] = t[1] + x.y;
        t[2] = t[2] + x.z;
        t[3] = t[3] + x.w;
        t[4] = t[4] + y.x;
        t[5] = t[5] + y.y;
        t[6] = t[6] + y.z;
        t[7] = t[7] + y.w;
      }
      finish<GBF16, MBF16>(a, id, col, t);
    }
  }
}

template <bool G, bool M>
cudaError_t launch_variant(const ApplyArgs& a, int num_sms, cudaStream_t stream) {
  static int blocks_per_sm = 0;  // the same for every device of one architecture
  if (blocks_per_sm == 0) {
    int b = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, apply_kernel<G, M>,
                                                                  kApplyThreads, 0);
    if (e != cudaSuccess) return e;
    blocks_per_sm = b > 0 ? b : 1;
  }
  apply_kernel<G, M><<<num_sms * blocks_per_sm, kApplyThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_apply(const ApplyArgs& a, int grad_bf16, int mg_bf16, int num_sms,
                         cudaStream_t stream) {
  if (grad_bf16) {
    return mg_bf16 ? launch_variant<true, true>(a, num_sms, stream)
                   : launch_variant<true, false>(a, num_sms, stream);
  }
  return mg_bf16 ? launch_variant<false, true>(a, num_sms, stream)
                 : launch_variant<false, false>(a, num_sms, stream);
}

}  // namespace ewg
