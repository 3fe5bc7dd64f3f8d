// SIMT kernels around the tensor-core steps: teacher-cache preparation, the merge of the
// per-vocabulary-tile statistics into lse and the per-position loss, the fixed-order loss
// sum, the split-K sum of dH, and the tf32 / bf16 copies of fp32 inputs.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "tc_gemm.cuh"

namespace fckl {

constexpr int PRE_WARPS = 4;
constexpr int K_LIMIT = 1024;
// Kernels that stream what a chunk's forward kept (the top-K builder's fp32 logits, the one
// call's fp16 e): threads per block, steps per thread, and the columns of one unit of
// topk_collect_kernel (one position, 8 columns per thread and step).
constexpr int GRAD_THREADS = 256;
constexpr int GRAD_STEPS = 4;
constexpr int GRAD_SEG = GRAD_THREADS * 8 * GRAD_STEPS;

// One warp per position of the chunk. Validates the teacher ids, orders the K slots by
// (id, slot) so the epilogues can walk them with a cursor, and forms p = exp(logp),
// S_n = sum_k p_nk and T_n = sum_k p_nk logp_nk (0 log 0 = 0). The cache holds the
// teacher's top-K log-probabilities without renormalisation, so S_n < 1.
__global__ void __launch_bounds__(32 * PRE_WARPS) preprocess_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ logp, int rows, int K, int V,
    int* __restrict__ sidx, float* __restrict__ sp, float* __restrict__ S, float* __restrict__ T,
    unsigned* __restrict__ status) {
  extern __shared__ int pre_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * PRE_WARPS + warp;
  if (row >= rows) return;  // warp-uniform; no block barrier below
  int* ids = pre_smem + warp * K;
  float* lps = reinterpret_cast<float*>(pre_smem + PRE_WARPS * K) + warp * K;
  const int32_t* ri = idx + static_cast<size_t>(row) * K;
  const float* rl = logp + static_cast<size_t>(row) * K;
  int bad = 0;
  for (int k = lane; k < K; k += 32) {
    const int i = ri[k];
    ids[k] = i;
    lps[k] = rl[k];
    bad |= (i < 0) | (i >= V);
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, ST_BAD_INDEX);
  __syncwarp();
  float s = 0.f, t = 0.f;
  for (int k = lane; k < K; k += 32) {
    const float lp = lps[k];
    const float pk = expf(lp);
    const int key = ids[k];
    int r = 0;
    for (int j = 0; j < K; ++j) {
      const int o = ids[j];
      r += (o < key) | ((o == key) & (j < k));
    }
    sidx[static_cast<size_t>(row) * K + r] = key;
    sp[static_cast<size_t>(row) * K + r] = pk;
    s += pk;
    t += (pk > 0.f) ? pk * lp : 0.f;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    t += __shfl_xor_sync(0xffffffffu, t, o);
  }
  if (lane == 0) {
    S[row] = s;
    T[row] = t;
  }
}

// Merge the (m, l, c) statistics of every vocabulary tile of a position:
//   lse_n  = M + log sum_t l_t exp(m_t - M),   c_n = sum_t c_t
//   loss_n = w_n (T_n - c_n + S_n lse_n)       (= w_n sum_k p_nk (logp_nk - z_{n,idx_nk} + lse_n))
// with w_n = 1 when no weights are given. 32 positions per block (lane = position, so each
// tile's statistics are read as one 128-byte line); COMBINE_WARPS warps split the tiles and are
// merged in a fixed order, so the result does not depend on timing. Many warps per block keep
// enough loads in flight: a chunk has only rows/32 blocks.
constexpr int COMBINE_WARPS = 32;
__global__ void __launch_bounds__(32 * COMBINE_WARPS) combine_kernel(
    const float* __restrict__ pm, const float* __restrict__ pl, const float* __restrict__ pc, int ld, int tiles,
    int rows, const float* __restrict__ S, const float* __restrict__ T, const float* __restrict__ weight,
    float* __restrict__ lse_out, float* __restrict__ loss_out) {
  __shared__ float sm[COMBINE_WARPS][32], sl[COMBINE_WARPS][32], sc[COMBINE_WARPS][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int row = blockIdx.x * 32 + lane;
  const bool valid = row < rows;
  float M = -INFINITY, Lr = 0.f, C = 0.f;
  if (valid) {
    // Batches of 8 tiles: the 24 loads of a batch are issued before any of them is merged.
    constexpr int B = 8;
    for (int t0 = w; t0 < tiles; t0 += COMBINE_WARPS * B) {
      float m[B], l[B], c[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int t = t0 + COMBINE_WARPS * b;
        const size_t o = static_cast<size_t>(t < tiles ? t : 0) * ld + row;
        m[b] = t < tiles ? pm[o] : -INFINITY;
        l[b] = t < tiles ? pl[o] : 0.f;
        c[b] = t < tiles ? pc[o] : 0.f;
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        if (m[b] == -INFINITY) continue;
        const float nm = fmaxf(M, m[b]);
        Lr = Lr * expf(M - nm) + l[b] * expf(m[b] - nm);
        M = nm;
        C += c[b];
      }
    }
  }
  sm[w][lane] = M;
  sl[w][lane] = Lr;
  sc[w][lane] = C;
  __syncthreads();
  if (w == 0 && valid) {
    for (int j = 1; j < COMBINE_WARPS; ++j) {
      const float m = sm[j][lane];
      if (m == -INFINITY) continue;
      const float nm = fmaxf(M, m);
      Lr = Lr * expf(M - nm) + sl[j][lane] * expf(m - nm);
      M = nm;
      C += sc[j][lane];
    }
    const float lse = M + logf(Lr);
    lse_out[row] = lse;
    const float wn = weight ? weight[row] : 1.f;
    loss_out[row] = wn * (T[row] - C + S[row] * lse);
  }
}

// Teacher cache builder, between the two passes over the vocabulary. R positions per block
// (R <= 8 keeps one position per warp in the search), 8 warps: lse_n from the per-tile (max, sum-exp) statistics, and the threshold
// thr_n = the K-th largest of the per-tile maxima (-inf when there are fewer tiles than K).
// The K largest tile maxima are K distinct logits of the row, so the row's K-th largest logit
// is >= thr_n and every top-K entry is at or above it. Also clears the candidate counters.
// Phase 1 reads the statistics coalesced across the block's rows (lane = row) and stages the
// maxima, as order-preserving integer keys, in shared memory [R][stride]; phase 2 runs a
// bitwise search for the K-th largest key, one warp per row. With `live` non-null the warp then
// lists, in tile order, the tiles whose maximum reaches the threshold (live[row][j], j <
// live_cnt[row]): only those can hold a candidate.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_key_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__global__ void __launch_bounds__(256) topk_threshold_kernel(const float* __restrict__ pm,
                                                             const float* __restrict__ pl, int ld, int tiles,
                                                             int rows, int R, int stride, int K,
                                                             float* __restrict__ lse_out,
                                                             float* __restrict__ thr_out, int* __restrict__ cnt,
                                                             int* __restrict__ live, int* __restrict__ live_cnt) {
  extern __shared__ uint32_t keys[];  // [R][stride]
  __shared__ float sm[8][32], sl[8][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int row = blockIdx.x * R + lane;
  const bool valid = lane < R && row < rows;
  float M = -INFINITY, Lr = 0.f;
  if (valid) {
    constexpr int B = 8;  // the loads of 8 tiles are issued before any of them is merged
    for (int t0 = w; t0 < tiles; t0 += 8 * B) {
      float m[B], l[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int t = t0 + 8 * b;
        const size_t o = static_cast<size_t>(t < tiles ? t : 0) * ld + row;
        m[b] = t < tiles ? pm[o] : -INFINITY;
        l[b] = t < tiles ? pl[o] : 0.f;
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int t = t0 + 8 * b;
        if (t >= tiles) continue;
        keys[lane * stride + t] = order_key(m[b]);
        const float nm = fmaxf(M, m[b]);
        Lr = Lr * expf(M - nm) + l[b] * expf(m[b] - nm);
        M = nm;
      }
    }
  }
  sm[w][lane] = M;
  sl[w][lane] = Lr;
  __syncthreads();
  if (w == 0 && valid) {
    for (int j = 1; j < 8; ++j) {
      const float m = sm[j][lane];
      if (m == -INFINITY) continue;
      const float nm = fmaxf(M, m);
      Lr = Lr * expf(M - nm) + sl[j][lane] * expf(m - nm);
      M = nm;
    }
    lse_out[row] = M + logf(Lr);
    cnt[row] = 0;
  }
  for (int r = w; r < R; r += 8) {  // warp-uniform rows
    const int row2 = blockIdx.x * R + r;
    if (row2 >= rows) break;
    float thr = -INFINITY;
    if (K <= tiles) {
      const uint32_t* kr = keys + r * stride;
      uint32_t prefix = 0;
      for (int bit = 31; bit >= 0; --bit) {
        const uint32_t cand = prefix | (1u << bit);
        int c = 0;
        for (int t = lane; t < tiles; t += 32) c += kr[t] >= cand;
        c = __reduce_add_sync(0xffffffffu, c);
        if (c >= K) prefix = cand;
      }
      thr = order_key_inv(prefix);
    }
    if (lane == 0) thr_out[row2] = thr;
    if (live) {  // tiles whose maximum is >= thr, i.e. whose key is >= prefix (all when thr = -inf)
      const uint32_t* kr = keys + r * stride;
      // keys order -0 below +0 but the comparison with the threshold does not: at a zero
      // threshold both zeros count
      const uint32_t kmin = K > tiles ? 0u : (thr == 0.f ? order_key(-0.f) : order_key(thr));
      int* lr = live + static_cast<int64_t>(row2) * tiles;
      int base = 0;
      for (int t0 = 0; t0 < tiles; t0 += 32) {
        const int t = t0 + lane;
        const bool on = t < tiles && kr[t] >= kmin;
        const uint32_t b = __ballot_sync(0xffffffffu, on);
        if (on) lr[base + __popc(b & ((1u << lane) - 1u))] = t;
        base += __popc(b);
      }
      if (lane == 0) live_cnt[row2] = base;
    }
  }
}

// Teacher cache builder, candidate collection from the logits pass 1 kept (fp32 Z, row pitch
// ld): every logit at or above the position's threshold is appended, with its token id, to
// the position's candidate list. Only the tiles the threshold kernel listed as live (tile
// maximum >= threshold; about K of a row's tiles) are read: a tile below it holds no
// candidate. The same values are compared with the same threshold as in the recomputing
// collect epilogue, so the candidate set is the same (the append order is not fixed in either;
// the select step orders the candidates fully). One warp per live tile (a lane takes 8 adjacent
// columns), each warp loading KC_BATCH tiles before comparing; the block's 8 warps share a
// position and blocks stride over positions.
constexpr int KC_BATCH = 4;

// BESIDE = true: the same code as a separate function, launched beside a tensor-core product
// with the largest shared-memory carve-out (as logit_grad_kernel<true>); it holds no shared
// memory, so one block fits beside a product CTA.
template <bool BESIDE>
__global__ void __launch_bounds__(256) topk_collect_kernel(
    const float* __restrict__ Z, int64_t ld, int rows, int V, int tiles, const float* __restrict__ thr,
    const int* __restrict__ live, const int* __restrict__ live_cnt, int* __restrict__ cnt,
    int* __restrict__ cand_v, float* __restrict__ cand_z, int cmax) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const float th = __ldg(thr + row);
    const int n = __ldg(live_cnt + row);
    const int* lr = live + static_cast<int64_t>(row) * tiles;
    const float* zr = Z + static_cast<int64_t>(row) * ld;
    for (int j0 = w * KC_BATCH; j0 < n; j0 += 8 * KC_BATCH) {
      float4 z[KC_BATCH][2];
      int cb[KC_BATCH];
#pragma unroll
      for (int b = 0; b < KC_BATCH; ++b) {
        const int j = j0 + b;
        cb[b] = j < n ? __ldg(lr + j) * VOCAB_TILE + 8 * lane : V;
        const int c = cb[b];
        if (c + 8 <= V) {
          z[b][0] = __ldcs(reinterpret_cast<const float4*>(zr + c));
          z[b][1] = __ldcs(reinterpret_cast<const float4*>(zr + c + 4));
        } else {
          float x[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) x[t] = c + t < V ? zr[c + t] : -INFINITY;
          z[b][0] = make_float4(x[0], x[1], x[2], x[3]);
          z[b][1] = make_float4(x[4], x[5], x[6], x[7]);
        }
      }
#pragma unroll
      for (int b = 0; b < KC_BATCH; ++b) {
        const int c = cb[b];
        const float x[8] = {z[b][0].x, z[b][0].y, z[b][0].z, z[b][0].w,
                            z[b][1].x, z[b][1].y, z[b][1].z, z[b][1].w};
        uint32_t hits = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) hits |= (x[t] >= th && c + t < V) ? (1u << t) : 0u;
        while (hits) {
          const int t = __ffs(hits) - 1;
          hits &= hits - 1;
          const int pos = atomicAdd(cnt + row, 1);
          if (pos < cmax) {
            float v = x[0];
#pragma unroll
            for (int q = 1; q < 8; ++q) v = (q == t) ? x[q] : v;
            cand_v[static_cast<int64_t>(row) * cmax + pos] = c + t;
            cand_z[static_cast<int64_t>(row) * cmax + pos] = v;
          }
        }
      }
    }
  }
}

// Teacher cache builder, last step. One warp per position: ranks the row's candidates by
// (logit descending, token id ascending) and writes the first K as (id, logit - lse).
// A row with more candidates than the buffer holds raises ST_CAPACITY (its output is then
// not the exact top-K).
// BESIDE: as for topk_collect_kernel (no shared memory either).
template <bool BESIDE>
__global__ void __launch_bounds__(128) topk_select_kernel(const int* __restrict__ cand_v,
                                                          const float* __restrict__ cand_z,
                                                          const int* __restrict__ cnt, int cmax, int rows, int K,
                                                          const float* __restrict__ lse,
                                                          int32_t* __restrict__ idx_out,
                                                          float* __restrict__ logp_out,
                                                          unsigned* __restrict__ status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + warp;
  if (row >= rows) return;  // warp-uniform
  int c = cnt[row];
  if (c > cmax) {
    if (lane == 0) atomicOr(status, ST_CAPACITY);
    c = cmax;
  }
  const int* cv = cand_v + static_cast<size_t>(row) * cmax;
  const float* cz = cand_z + static_cast<size_t>(row) * cmax;
  const float l = lse[row];
  for (int i = lane; i < c; i += 32) {
    const float zi = cz[i];
    const int vi = cv[i];
    int r = 0;
    for (int j = 0; j < c; ++j) {
      const float zj = cz[j];
      const int vj = cv[j];
      r += (zj > zi) | ((zj == zi) & (vj < vi));
    }
    if (r < K) {
      idx_out[static_cast<size_t>(row) * K + r] = vi;
      logp_out[static_cast<size_t>(row) * K + r] = zi - l;
    }
  }
}

// Sum of the per-position losses in a fixed order, in fp64.
__global__ void __launch_bounds__(1024) loss_reduce_kernel(const float* __restrict__ row_loss, int64_t n,
                                                           float* __restrict__ loss) {
  __shared__ double sh[1024];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += 1024) s += static_cast<double>(row_loss[i]);
  sh[threadIdx.x] = s;
  __syncthreads();
  for (int o = 512; o > 0; o >>= 1) {
    if (threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = static_cast<float>(sh[0]);
}

__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
  uint2 u;
  u.x = pack_bf16x2(v.x, v.y);
  u.y = pack_bf16x2(v.z, v.w);
  *reinterpret_cast<uint2*>(p) = u;
}

// dH[row] = sum over K-splits of the fp32 partial products, in split order, stored in
// the type of H. part is [splits][split_rows][d]; d % 4 == 0.
template <typename OutT>
__global__ void __launch_bounds__(256) dh_reduce_kernel(const float* __restrict__ part, int splits,
                                                        int64_t split_stride, int rows, int d,
                                                        OutT* __restrict__ out) {
  const int64_t n4 = static_cast<int64_t>(rows) * d / 4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i * 4;
    float4 a = *reinterpret_cast<const float4*>(part + e);
    for (int s = 1; s < splits; ++s) {
      const float4 b = *reinterpret_cast<const float4*>(part + s * split_stride + e);
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    store4(out + e, a);
  }
}

// G, in place, from what the forward kept of the chunk's logits: the slab G holds
// e = exp(z - m) as fp16 (EPI_FWD_KEEP), m being the logit's tile maximum (pm, one per row and
// vocabulary tile). Each element becomes G = f * e - scale * w_n * p at the cached ids, with
// f = scale * w_n * S_n * exp(m - lse_n), rounded to bf16 and written over e: the same
// operations in the same order as the EPI_LOGIT_GRAD epilogue, so G is bitwise the one the
// recomputing path forms. HBM-bound (4 bytes per element: 2 read, 2 written); a unit is one
// position and KG_SEG columns, each thread takes 16 adjacent columns per step (two 16-byte
// loads and stores at the same addresses), GRAD_STEPS steps 4096 columns apart, all loads
// issued before the arithmetic (128 bytes in flight per thread), together with the steps' tile
// maxima and the row's scalars. Each thread walks the row's ordered cache slots with one
// cursor, read through L1 (no shared memory: a block then fits on an SM beside a tensor-core
// product that holds nearly all of it, so this pass can run concurrently with one). Row pitch
// ld is a multiple of 8 elements; columns in [V, ld) are written as 0.
constexpr int KG_COLS = 16;
constexpr int KG_SEG = GRAD_THREADS * KG_COLS * GRAD_STEPS;

// BESIDE = true: the same code as a separate function, launched beside a tensor-core product
// and set to prefer the largest shared-memory carve-out, so that an SM it lands on first stays
// configured for that product's CTAs; BESIDE = false keeps the default carve-out (more L1 for
// loads in flight) for the pass that runs alone.
template <bool BESIDE>
__global__ void __launch_bounds__(GRAD_THREADS) logit_grad_kernel(
    __nv_bfloat16* __restrict__ G, int64_t ld, int rows, int V, int K, const int* __restrict__ sidx,
    const float* __restrict__ sp, const float* __restrict__ S, const float* __restrict__ lse,
    const float* __restrict__ wrow, float gscale, const float* __restrict__ pm, int ld_part) {
  const int segs = (V + KG_SEG - 1) / KG_SEG;
  const int64_t units = static_cast<int64_t>(rows) * segs;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int row = static_cast<int>(u / segs);
    const int seg = static_cast<int>(u - static_cast<int64_t>(row) * segs);
    __nv_bfloat16* gr = G + static_cast<int64_t>(row) * ld;
    const int c0 = seg * KG_SEG + KG_COLS * static_cast<int>(threadIdx.x);
    // everything the unit reads is requested first: e, the tile maxima, the row's scalars
    uint4 e[2 * GRAD_STEPS];
    float mt[GRAD_STEPS];
#pragma unroll
    for (int i = 0; i < GRAD_STEPS; ++i) {
      const int c = c0 + i * GRAD_THREADS * KG_COLS;
      // 8-column halves wholly past V are not read (the row pitch ends at a multiple of 8)
      e[2 * i] = c < V ? *reinterpret_cast<const uint4*>(gr + c) : make_uint4(0u, 0u, 0u, 0u);
      e[2 * i + 1] = c + 8 < V ? *reinterpret_cast<const uint4*>(gr + c + 8) : make_uint4(0u, 0u, 0u, 0u);
      mt[i] = c < V ? __ldg(pm + static_cast<int64_t>(c / VOCAB_TILE) * ld_part + row) : 0.f;
    }
    const float wv = wrow ? __ldg(wrow + row) : 1.f;
    const float sv = __ldg(S + row), lv = __ldg(lse + row);
    const int* ids = sidx + static_cast<int64_t>(row) * K;
    const float* pv = sp + static_cast<int64_t>(row) * K;
    const float gs = __fmul_rn(gscale, wv);
    const float a = __fmul_rn(gs, sv);
    const float nl = __fmul_rn(-lv, LOG2E);
    int lo = 0, hi = K;  // cursor: first slot whose id is >= c0
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(ids + mid) < c0)
        lo = mid + 1;
      else
        hi = mid;
    }
    int k = lo;
#pragma unroll
    for (int i = 0; i < GRAD_STEPS; ++i) {
      const int c = c0 + i * GRAD_THREADS * KG_COLS;
      if (c >= V) break;
      const float f = tile_factor(a, mt[i], nl);
      const __half* eh = reinterpret_cast<const __half*>(&e[2 * i]);
      float x[KG_COLS];
#pragma unroll
      for (int t = 0; t < KG_COLS; ++t) x[t] = grad_dense(f, eh[t]);
      while (k < K && __ldg(ids + k) < c) ++k;
      while (k < K && __ldg(ids + k) < c + KG_COLS) {
        const int pos = __ldg(ids + k) - c;
        const float v = __fmul_rn(gs, __ldg(pv + k));
#pragma unroll
        for (int t = 0; t < KG_COLS; ++t) x[t] = (t == pos) ? __fsub_rn(x[t], v) : x[t];
        ++k;
      }
      if (c + KG_COLS > V) {
#pragma unroll
        for (int t = 0; t < KG_COLS; ++t) x[t] = c + t < V ? x[t] : 0.f;
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (c + 8 * hh >= V) break;
        uint4 w;
        w.x = pack_bf16x2(x[8 * hh + 0], x[8 * hh + 1]);
        w.y = pack_bf16x2(x[8 * hh + 2], x[8 * hh + 3]);
        w.z = pack_bf16x2(x[8 * hh + 4], x[8 * hh + 5]);
        w.w = pack_bf16x2(x[8 * hh + 6], x[8 * hh + 7]);
        *reinterpret_cast<uint4*>(gr + c + 8 * hh) = w;
      }
    }
  }
}

// fp32 -> tf32 (10 explicit mantissa bits, round to nearest with ties away from zero), kept
// in an fp32 container with the low 13 bits zero: the value the tf32 tensor-core products
// then read exactly (they would otherwise drop the low bits, a bias toward zero).
__device__ __forceinline__ float round_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// fp32 inputs, one read: tf32-rounded copy into t32 and/or bf16 copy (round to nearest even)
// into b16 (either may be null); n % 4 == 0.
__global__ void __launch_bounds__(256) cvt_inputs_kernel(const float* __restrict__ src, float* __restrict__ t32,
                                                         __nv_bfloat16* __restrict__ b16, int64_t n) {
  const int64_t n4 = n / 4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = *reinterpret_cast<const float4*>(src + 4 * i);
    if (t32)
      *reinterpret_cast<float4*>(t32 + 4 * i) =
          make_float4(round_tf32(v.x), round_tf32(v.y), round_tf32(v.z), round_tf32(v.w));
    if (b16) store4(b16 + 4 * i, v);
  }
}

}  // namespace fckl
