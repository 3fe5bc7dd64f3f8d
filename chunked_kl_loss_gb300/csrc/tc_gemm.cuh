// Persistent, warp-specialised tcgen05 GEMM engine for the fused chunked KL loss.
//
// One CTA per SM, 192 threads. With CG = 2 two SMs of a cluster form a pair that computes a
// 256 x BN tile with tcgen05.mma.cta_group::2: each CTA stages its 128 rows of A and half of
// B, the even CTA issues the MMAs, and each CTA's TMEM receives its 128 rows of the result
// (CG = 1: one CTA per 128 x BN tile). K-blocks of 64 bf16 (32 fp32), two per ring stage in
// the bf16 logits products.
//   warp 0     : TMA producer (one lane) filling a shared-memory ring (192 KB per CTA for pairs)
//   warp 1     : TMEM owner and, in the even CTA, MMA issuer (one lane); two TMEM
//                accumulators of 128 x 256 fp32 per CTA so the epilogue of one tile
//                overlaps the main loop of the next
//   warps 2..5 : epilogue, one TMEM lane quarter (32 rows) each
// Work units (tile, K-split) are dealt round-robin over the persistent CTAs in an order
// chosen by the host so that concurrently running CTAs share operand tiles in L2.
//
// Epilogues (the steps of the method that follow each projection):
//   EPI_FWD_STATS : per row, the tile's maximum m over its vocabulary columns (first pass
//                   over the accumulator), the gather of the logits at the teacher's cached
//                   ids, and sum_v exp(z_v - m) (second pass); writes one (m, l, c) triple per
//                   row and vocabulary tile ("Fused, chunked KL loss": fold the chunk's
//                   logits into the running loss, then drop them)
//   EPI_FWD_KEEP  : EPI_FWD_STATS that also stores e = exp(z - m) as fp16 with TMA into the
//                   chunk's gradient slab, so that the chunk's backward can form G from it
//                   in place instead of recomputing the logits
//   EPI_FWD_Z     : EPI_FWD_STATS that also stores the fp32 logits with TMA (teacher top-K
//                   builder: its second pass compares exact logits)
//   EPI_LOGIT_GRAD: G = scale * w_n * (S_n exp(z - lse_n) - p at the cached ids), rounded
//                   to bf16 and stored with TMA (the backward pass recomputes the chunk);
//                   exp(z - lse_n) is formed as exp(m - lse_n) * fp16(exp(z - m)) with the
//                   tile maximum m, the same values the EPI_FWD_KEEP path keeps
//   EPI_STORE_F32 : fp32 tile stored, or reduce-added, with TMA (dH partials, dW)
//   EPI_TOPK_COLLECT: appends every logit at or above the row's threshold, with its token
//                   id, to the row's candidate list (teacher top-K cache builder)
// Every wait is bounded by WAIT_TIMEOUT_NS; on expiry the CTA records FCKL status bit
// ST_TIMEOUT, lets its copies and MMAs in flight drain, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <climits>
#include <cstdint>

#include "ptx.cuh"

namespace fckl {

constexpr int BM = 128;  // rows of A per CTA
constexpr int BK = 64;   // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int VOCAB_TILE = 256;  // vocabulary columns per tile of the logits kernels (their BN)
constexpr int EPI_WARPS = 4;
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_STRIDE = 256;  // TMEM column offset of the second accumulator
constexpr uint32_t EPI_BUF_BYTES = 4096;  // 32 rows x 128 B staging box per epilogue warp
constexpr uint64_t WAIT_TIMEOUT_NS = 2000000000ull;
constexpr float LOG2E = 1.4426950408889634f;

enum : unsigned { ST_BAD_INDEX = 1u, ST_TIMEOUT = 2u, ST_CAPACITY = 4u };
enum { EPI_FWD_STATS = 0, EPI_LOGIT_GRAD = 1, EPI_STORE_F32 = 2, EPI_TOPK_COLLECT = 3, EPI_FWD_KEEP = 4, EPI_FWD_Z = 5 };

struct Sched {
  int m_blocks, n_blocks, k_blocks;
  int splits, kb_per_split;
  int n_outer;  // 1: unit order is (split, n, m) with m fastest; 0: (split, m, n) with n fastest
};

struct TcParams {
  CUtensorMap tmA;  // operand A (M x K)
  CUtensorMap tmB;  // operand B (N x K)
  CUtensorMap tmC;  // epilogue output
  CUtensorMap tmP;  // epilogue output, unswizzled 128-row x 256-column boxes for L2 prefetch
  Sched sch;
  int num_units;
  unsigned* status;
  // logits epilogues
  int rows_valid, V, K;
  const int* sidx;   // [rows][K] teacher ids of the chunk, ascending per row
  const float* sp;   // [rows][K] matching teacher probabilities
  const float* S;    // [rows] kept teacher mass
  const float* lse;  // [rows] log-partition (backward)
  const float* wrow;  // [rows] position weights, or null for all ones (backward)
  float gscale;
  float* pm;
  float* pl;
  float* pc;
  int ld_part;
  // fp32 store epilogue
  int c_split_rows;  // rows between the slabs of successive K-splits in tmC
  int c_reduce;      // 1: reduce-add into tmC, 0: plain store
  int c_xlim, c_ylim;  // extent of tmC: boxes starting at or past it are not issued
  int c_prefetch;      // 1: prefetch each unit's output tile into L2 when its loads start
  // 1 when tmA / tmB is a 3-D map that fetches a whole stage of the operand in one copy: for an
  // MN-major operand (64 MN-values, K rows, 64-wide MN blocks), instead of one 2-D copy per block;
  int a_3d, b_3d;  // (bf16 products, two K-blocks per stage) also for K-major operands: one 3-D
                   // copy (64 K-values, rows, K-blocks) fetches a stage's two K-blocks
  // top-K candidate collection (teacher cache builder)
  const float* thr;  // [rows] logits at or above it are candidates
  int* cnt;          // [rows] candidates found (may exceed cmax)
  int* cand_v;       // [rows][cmax] token ids
  float* cand_z;     // [rows][cmax] logits
  int cmax;
};

// Shared-memory layout of one CTA. CG = CTAs per MMA (1: a 128 x BN tile per CTA; 2: a
// 256 x BN tile per CTA pair, each CTA holding its 128 rows of A and BN/2 rows of B). A ring
// stage holds KPS K-blocks (128 bytes of K per row each): the same bytes in flight in fewer,
// larger stages, so that the per-stage hand-off (barriers, commit, copies) is paid less often.
template <int CG, int BN, int KPS>
struct TcSmem {
  static constexpr int STAGES = (CG == 2 ? 6 : 4) / KPS;
  static constexpr int BN_CTA = BN / CG;
  static constexpr uint32_t A_KB = BM * BK * 2;      // one K-block of A
  static constexpr uint32_t B_KB = BN_CTA * BK * 2;  // one K-block of B
  static constexpr uint32_t A_BYTES = KPS * A_KB;
  static constexpr uint32_t B_BYTES = KPS * B_KB;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t EPI_OFF = STAGES * STAGE_BYTES;
  static constexpr uint32_t BAR_OFF = EPI_OFF + EPI_WARPS * 2 * EPI_BUF_BYTES;
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 2 + 2 + 1;
  static constexpr uint32_t END = BAR_OFF + NUM_BARS * 8 + 16;
  static constexpr uint32_t DYN_BYTES = END + 1024;  // slack for 1024-byte alignment
};

__device__ __forceinline__ void decode_unit(const Sched& s, int u, int& mb, int& nb, int& sp, int& kb0,
                                            int& kb1) {
  const int tiles = s.m_blocks * s.n_blocks;
  sp = u / tiles;
  const int r = u - sp * tiles;
  if (s.n_outer) {
    nb = r / s.m_blocks;
    mb = r - nb * s.m_blocks;
  } else {
    mb = r / s.n_blocks;
    nb = r - mb * s.n_blocks;
  }
  kb0 = sp * s.kb_per_split;
  kb1 = min(s.k_blocks, kb0 + s.kb_per_split);
}

// Bounded wait on one mbarrier phase, polled by the calling thread. Returns false when the
// CTA is aborting (another role gave up) or when the deadline passed (then it also raises
// the abort flag and the status bit).
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned* status, uint64_t timeout_ns = WAIT_TIMEOUT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        atomicOr(status, ST_TIMEOUT);
        return false;
      }
    }
  }
}

// Same, for teardown: ignores the abort flag, still bounded.
__device__ __forceinline__ bool drain_phase(uint64_t* bar, uint32_t parity, unsigned* status) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 31u && globaltimer_ns() - t0 > WAIT_TIMEOUT_NS) {
      atomicOr(status, ST_TIMEOUT);
      return false;
    }
  }
}

// Warp-uniform wait: lane 0 polls, the verdict is broadcast.
__device__ __forceinline__ bool warp_wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                unsigned* status) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_phase(bar, parity, abort_flag, status) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// First slot k of a row's ascending id list with ids[k] >= key.
__device__ __forceinline__ int lower_bound_ids(const int* ids, int n, int key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(ids + mid) < key)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

// x[pos] for a runtime pos in [0, 32) without leaving registers.
__device__ __forceinline__ float pick32(const float (&x)[32], int pos) {
  float r = 0.f;
#pragma unroll
  for (int t = 0; t < 32; ++t) r = (t == pos) ? x[t] : r;
  return r;
}
__device__ __forceinline__ void sub32(float (&x)[32], int pos, float v) {
#pragma unroll
  for (int t = 0; t < 32; ++t) x[t] = (t == pos) ? __fsub_rn(x[t], v) : x[t];
}

// The dense part of G, in steps that every path takes identically (each operation rounded
// on its own, no contraction into FMAs), so that G formed from the kept values has the bits
// of G formed from recomputed logits. With the tile maximum m (ml = m * log2(e)):
//   e = exp(z - m), kept as fp16 (relative rounding 2^-11, finer than G's own bf16 2^-9)
//   f = a * exp(m - lse_n),  a = scale * w_n * S_n,  nl = -lse_n * log2(e)
//   G_dense = f * e
__device__ __forceinline__ float exp_in_tile(float z, float ml) { return ex2_approx(fmaf(z, LOG2E, -ml)); }
__device__ __forceinline__ float tile_factor(float a, float m, float nl) {
  return __fmul_rn(a, ex2_approx(fmaf(m, LOG2E, nl)));
}
__device__ __forceinline__ float grad_dense(float f, __half e) { return __fmul_rn(f, __half2float(e)); }
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float max32(const float (&x)[32]) {
  float m = x[0];
#pragma unroll
  for (int t = 1; t < 32; ++t) m = fmaxf(m, x[t]);
  return m;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Self-test of the bounded wait: one thread waits on a barrier that nothing arrives at; the
// wait gives up after timeout_ns, records ST_TIMEOUT and the kernel returns normally.
__global__ void wait_timeout_selftest_kernel(unsigned* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_phase(&bar, 0, &abort_flag, status, timeout_ns);
}

// Bounded wait whose acquire also covers arrivals from the peer CTA of a pair.
__device__ __forceinline__ bool wait_phase_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                   unsigned* status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 31u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > WAIT_TIMEOUT_NS) {
        *abort_flag = 1;
        atomicOr(status, ST_TIMEOUT);
        return false;
      }
    }
  }
}

// TF32: the operands are fp32 and the MMAs run as kind::tf32 (both operands K-major). A stage
// then holds 32 fp32 values of K per row: the same 128 bytes, the same swizzled layout and the
// same descriptors as 64 bf16 values, with four MMAs of K = 8 instead of K = 16.
template <int CG, int BN, bool A_MN, bool B_MN, int EPI, bool TF32 = false>
__global__ void __launch_bounds__(NUM_THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  // K-blocks per ring stage: two for the bf16 products with both operands K-major (the logits
  // products), where the larger stages measured 4-6% faster; one for dH and dW, where they did
  // not help (dW, both operands MN-major, was 6% slower).
  constexpr int KPS = (TF32 || A_MN || B_MN) ? 1 : 2;
  using L = TcSmem<CG, BN, KPS>;
  constexpr int NST = L::STAGES;
  constexpr int BN_CTA = L::BN_CTA;
  constexpr int KE = TF32 ? BK / 2 : BK;  // K elements per K-block (128 bytes of each row)
  static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair per MMA");
  static_assert(!B_MN || BN_CTA % 64 == 0, "MN-major B is staged in 64-wide blocks");
  static_assert(!TF32 || (!A_MN && !B_MN), "tf32 operands are staged K-major");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + NST;
  uint64_t* tfull = empty + NST;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;  // position in the CTA pair
  const bool leader = rank == 0;
  const int cluster_id = blockIdx.x / CG;
  const int num_clusters = gridDim.x / CG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], EPI_WARPS * CG);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&p.tmA);
    prefetch_tmap(&p.tmB);
    if (EPI != EPI_FWD_STATS) prefetch_tmap(&p.tmC);
  }
  if (warp == 1) {
    if constexpr (CG == 2) {
      tmem_alloc_pair(tmem_holder, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // the peer's barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (each CTA)
    if (lane == 0) {
      uint32_t cnt = 0;
      uint32_t armed = 0, armed_par = 0;  // per stage: ever armed, parity of the last arming
      bool ok = true;
      const uint32_t full_base = CG == 2 ? mapa_shared(smem_u32(full), 0) : smem_u32(full);
      for (int u = cluster_id; ok && u < p.num_units; u += num_clusters) {
        int mb, nb, sp, kb0, kb1;
        decode_unit(p.sch, u, mb, nb, sp, kb0, kb1);
        const int arow = mb * BM * CG + static_cast<int>(rank) * BM;       // this CTA's A rows
        const int bcol = nb * BN + static_cast<int>(rank) * BN_CTA;        // this CTA's B rows/cols
        // A reduce-add epilogue reads its output tile back from memory: start that read now,
        // a whole main loop before the epilogue needs it.
        if (EPI == EPI_STORE_F32 && p.c_prefetch && nb * BN < p.c_xlim && arow < p.c_ylim)
          tma_prefetch_l2_2d(&p.tmP, nb * BN, arow);
        for (int kb = kb0; kb < kb1; kb += KPS, ++cnt) {
          const uint32_t s = cnt % NST, ph = (cnt / NST) & 1u;
          if (!wait_phase(&empty[s], ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(&full[s], CG * L::STAGE_BYTES);
            armed |= 1u << s;
            armed_par = (armed_par & ~(1u << s)) | (ph << s);
          }
          uint8_t* a = smem + s * L::STAGE_BYTES;
          uint8_t* b = a + L::A_BYTES;
          const uint32_t fb = full_base + s * 8u;
          auto load = [&](void* dst, const CUtensorMap* m, int x, int y) {
            if constexpr (CG == 2)
              tma_load_2d_pair(dst, m, fb, x, y);
            else
              tma_load_2d(dst, m, &full[s], x, y);
          };
          // Stage layouts, as the 3-D boxes lay them out. K-major: K-block j of the stage at
          // j * A_KB (rows x 128 bytes). MN-major: the 64-wide MN block i at i * KPS * 8192, its
          // KPS * 64 K rows in order, so K-block j starts j * 8192 bytes into each block. A copy
          // past the unit's K range (an odd count) or past K lands data the MMAs skip or zeros.
          if (!A_MN) {
            if (!TF32 && CG == 2 && p.a_3d) {
              tma_load_3d_pair(a, &p.tmA, fb, 0, arow, kb);
            } else {
#pragma unroll
              for (int j = 0; j < KPS; ++j) load(a + j * L::A_KB, &p.tmA, (kb + j) * KE, arow);
            }
          } else if (CG == 2 && p.a_3d) {
            tma_load_3d_pair(a, &p.tmA, fb, 0, kb * BK, arow / 64);
          } else {
#pragma unroll
            for (int i = 0; i < BM / 64; ++i) load(a + i * KPS * 8192, &p.tmA, arow + 64 * i, kb * BK);
          }
          if (!B_MN) {
            if (!TF32 && CG == 2 && p.b_3d) {
              tma_load_3d_pair(b, &p.tmB, fb, 0, bcol, kb);
            } else {
#pragma unroll
              for (int j = 0; j < KPS; ++j) load(b + j * L::B_KB, &p.tmB, (kb + j) * KE, bcol);
            }
          } else if (CG == 2 && p.b_3d) {
            tma_load_3d_pair(b, &p.tmB, fb, 0, kb * BK, bcol / 64);
          } else {
#pragma unroll
            for (int i = 0; i < BN_CTA / 64; ++i) load(b + i * KPS * 8192, &p.tmB, bcol + 64 * i, kb * BK);
          }
        }
      }
      // Every copy this pair started must land before a CTA may exit. The leader's full
      // barriers count both CTAs' bytes; a peer that gave up early waits a little for its
      // own copies, whose barrier it cannot poll.
      if (leader) {
        for (int s = 0; s < NST; ++s)
          if (armed & (1u << s)) drain_phase(&full[s], (armed_par >> s) & 1u, p.status);
      } else if (!ok) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA)
    if (lane == 0 && leader) {
      constexpr uint32_t IDESC = TF32 ? make_idesc_tf32(BM * CG, BN) : make_idesc_bf16(BM * CG, BN, A_MN, B_MN);
      uint32_t cnt = 0, it = 0;
      bool ok = true;
      for (int u = cluster_id; ok && u < p.num_units; u += num_clusters, ++it) {
        int mb, nb, sp, kb0, kb1;
        decode_unit(p.sch, u, mb, nb, sp, kb0, kb1);
        const uint32_t acc = it & 1u, use = it >> 1;
        const bool got = CG == 2 ? wait_phase_cluster(&tempty[acc], (use & 1u) ^ 1u, abort_flag, p.status)
                                 : wait_phase(&tempty[acc], (use & 1u) ^ 1u, abort_flag, p.status);
        if (!got) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_STRIDE;
        for (int kb = kb0; kb < kb1; kb += KPS, ++cnt) {
          const uint32_t s = cnt % NST, ph = (cnt / NST) & 1u;
          if (!wait_phase(&full[s], ph, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + s * L::STAGE_BYTES);
          const uint32_t b_addr = a_addr + L::A_BYTES;
#pragma unroll
          for (int q = 0; q < KPS * (BK / 16); ++q) {
            const int j = q / (BK / 16), kk = q % (BK / 16);  // K-block of the stage, K step in it
            if (KPS > 1 && kb + j >= kb1) break;               // past the unit's K range
            const uint64_t ad = A_MN ? make_sdesc_sw128(a_addr + j * 8192 + kk * 2048, KPS * 8192, 1024)
                                     : make_sdesc_sw128(a_addr + j * L::A_KB + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? make_sdesc_sw128(b_addr + j * 8192 + kk * 2048, KPS * 8192, 1024)
                                     : make_sdesc_sw128(b_addr + j * L::B_KB + kk * 32, 16, 1024);
            const uint32_t accum = (kb > kb0 || q > 0) ? 1u : 0u;
            if constexpr (CG == 2 && TF32)
              umma_tf32_pair(d_tmem, ad, bd, IDESC, accum);
            else if constexpr (CG == 2)
              umma_bf16_pair(d_tmem, ad, bd, IDESC, accum);
            else if constexpr (TF32)
              umma_tf32(d_tmem, ad, bd, IDESC, accum);
            else
              umma_bf16(d_tmem, ad, bd, IDESC, accum);
          }
          if constexpr (CG == 2)
            umma_commit_pair(&empty[s], 0x3);
          else
            umma_commit(&empty[s]);
        }
        if (!ok) break;
        if constexpr (CG == 2)
          umma_commit_pair(&tfull[acc], 0x3);
        else
          umma_commit(&tfull[acc]);
      }
      // All MMAs issued by this thread must finish before TMEM is released.
      if constexpr (CG == 2)
        umma_commit_pair(drain, 0x1);
      else
        umma_commit(drain);
      drain_phase(drain, 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue (each CTA)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t* ebuf0 = smem + L::EPI_OFF + (warp - 2) * 2 * EPI_BUF_BYTES;
    const uint32_t tempty_leader = CG == 2 ? mapa_shared(smem_u32(tempty), 0) : 0u;
    auto release_acc = [&](uint32_t acc) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CG == 2 && !leader)
          mbar_arrive_cluster(tempty_leader + acc * 8u);
        else
          mbar_arrive(&tempty[acc]);
      }
    };
    uint32_t it = 0, ecnt = 0;
    for (int u = cluster_id; u < p.num_units; u += num_clusters, ++it) {
      int mb, nb, sp, kb0, kb1;
      decode_unit(p.sch, u, mb, nb, sp, kb0, kb1);
      const uint32_t acc = it & 1u, use = it >> 1;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + acc * ACC_STRIDE;
      const int row0 = mb * BM * CG + static_cast<int>(rank) * BM + 32 * q;  // first row of this warp
      const int row = row0 + lane;

      if constexpr (EPI == EPI_FWD_STATS || EPI == EPI_FWD_KEEP || EPI == EPI_FWD_Z || EPI == EPI_LOGIT_GRAD) {
        const bool valid = row < p.rows_valid;
        const int v0 = nb * BN;
        const int* ids = p.sidx + static_cast<size_t>(valid ? row : 0) * p.K;
        const float* pr = p.sp + static_cast<size_t>(valid ? row : 0) * p.K;
        int k = p.K, nxt = INT_MAX;
        if (valid) {
          k = lower_bound_ids(ids, p.K, v0);
          nxt = k < p.K ? __ldg(ids + k) : INT_MAX;
        }
        if constexpr (EPI == EPI_FWD_STATS || EPI == EPI_FWD_KEEP || EPI == EPI_FWD_Z) {
          if (!warp_wait_phase(&tfull[acc], use & 1u, abort_flag, p.status)) break;
          tc_fence_after();
          // pass 1: the tile maximum (columns past V excluded) and the gathered sum
          float m = -INFINITY, c = 0.f;
#pragma unroll 1
          for (int j = 0; j < BN / 32; ++j) {
            float x[32];
            __syncwarp();
            tmem_ld32(taddr + 32 * j, x);
            const int cb = v0 + 32 * j;
            if constexpr (EPI == EPI_FWD_Z) {
              // stage the raw logits (32 rows x 32 columns, 128-byte swizzle) and store them
              uint8_t* buf = ebuf0 + (ecnt & 1u) * EPI_BUF_BYTES;
              if (ecnt >= 2 && lane == 0) bulk_wait_read<1>();
              __syncwarp();
#pragma unroll
              for (int cc = 0; cc < 8; ++cc) {
                const int chunk16 = cc ^ (lane & 7);
                *reinterpret_cast<float4*>(buf + lane * 128 + chunk16 * 16) =
                    make_float4(x[4 * cc + 0], x[4 * cc + 1], x[4 * cc + 2], x[4 * cc + 3]);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                if (cb < p.c_xlim && row0 < p.c_ylim) tma_store_2d(&p.tmC, buf, cb, row0);
                bulk_commit();
              }
              ++ecnt;
            }
            if (cb + 32 > p.V) {
#pragma unroll
              for (int t = 0; t < 32; ++t)
                if (cb + t >= p.V) x[t] = -INFINITY;
            }
            while (nxt < cb + 32) {
              c = fmaf(__ldg(pr + k), pick32(x, nxt - cb), c);
              ++k;
              nxt = k < p.K ? __ldg(ids + k) : INT_MAX;
            }
            m = fmaxf(m, max32(x));
          }
          // pass 2: sum of exp(z - m); EPI_FWD_KEEP also stores fp16 exp(z - m), 64-column boxes
          const float ml = __fmul_rn(m, LOG2E);
          float l = 0.f;
#pragma unroll 1
          for (int jj = 0; jj < BN / 64; ++jj) {
            uint8_t* buf = ebuf0 + (ecnt & 1u) * EPI_BUF_BYTES;
            if constexpr (EPI == EPI_FWD_KEEP) {
              if (ecnt >= 2 && lane == 0) bulk_wait_read<1>();
              __syncwarp();
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int j = 2 * jj + h;
              float x[32];
              __syncwarp();
              tmem_ld32(taddr + 32 * j, x);
              if (j == BN / 32 - 1) release_acc(acc);
              const int cb = v0 + 32 * j;
              if (cb + 32 > p.V) {
#pragma unroll
                for (int t = 0; t < 32; ++t)
                  if (cb + t >= p.V) x[t] = -INFINITY;
              }
#pragma unroll
              for (int t = 0; t < 32; ++t) {
                x[t] = exp_in_tile(x[t], ml);
                l += x[t];
              }
              if constexpr (EPI == EPI_FWD_KEEP) {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                  uint4 w;
                  w.x = pack_f16x2(x[8 * cc + 0], x[8 * cc + 1]);
                  w.y = pack_f16x2(x[8 * cc + 2], x[8 * cc + 3]);
                  w.z = pack_f16x2(x[8 * cc + 4], x[8 * cc + 5]);
                  w.w = pack_f16x2(x[8 * cc + 6], x[8 * cc + 7]);
                  const int chunk16 = (4 * h + cc) ^ (lane & 7);
                  *reinterpret_cast<uint4*>(buf + lane * 128 + chunk16 * 16) = w;
                }
              }
            }
            if constexpr (EPI == EPI_FWD_KEEP) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                const int sx = v0 + 64 * jj;
                if (sx < p.c_xlim && row0 < p.c_ylim) tma_store_2d(&p.tmC, buf, sx, row0);
                bulk_commit();
              }
              ++ecnt;
            }
          }
          if (valid) {
            const size_t o = static_cast<size_t>(nb) * p.ld_part + row;
            p.pm[o] = m;
            p.pl[o] = l;
            p.pc[o] = c;
          }
        } else {
          const float gs = valid ? __fmul_rn(p.gscale, p.wrow ? __ldg(p.wrow + row) : 1.f) : 0.f;
          const float a = __fmul_rn(gs, valid ? __ldg(p.S + row) : 0.f);
          const float nl = valid ? __fmul_rn(-__ldg(p.lse + row), LOG2E) : 0.f;
          if (!warp_wait_phase(&tfull[acc], use & 1u, abort_flag, p.status)) break;
          tc_fence_after();
          // pass 1: the tile maximum, as the forward took it
          float m = -INFINITY;
#pragma unroll 1
          for (int j = 0; j < BN / 32; ++j) {
            float x[32];
            __syncwarp();
            tmem_ld32(taddr + 32 * j, x);
            const int cb = v0 + 32 * j;
            if (cb + 32 > p.V) {
#pragma unroll
              for (int t = 0; t < 32; ++t)
                if (cb + t >= p.V) x[t] = -INFINITY;
            }
            m = fmaxf(m, max32(x));
          }
          const float ml = __fmul_rn(m, LOG2E);
          const float f = tile_factor(a, m, nl);
#pragma unroll 1
          for (int jj = 0; jj < BN / 64; ++jj, ++ecnt) {
            uint8_t* buf = ebuf0 + (ecnt & 1u) * EPI_BUF_BYTES;
            if (ecnt >= 2 && lane == 0) bulk_wait_read<1>();
            __syncwarp();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int j = 2 * jj + h;
              float x[32];
              __syncwarp();
              tmem_ld32(taddr + 32 * j, x);
              if (j == BN / 32 - 1) release_acc(acc);
              const int cb = v0 + 32 * j;
#pragma unroll
              for (int t = 0; t < 32; ++t) x[t] = grad_dense(f, __float2half_rn(exp_in_tile(x[t], ml)));
              while (nxt < cb + 32) {
                sub32(x, nxt - cb, __fmul_rn(gs, __ldg(pr + k)));
                ++k;
                nxt = k < p.K ? __ldg(ids + k) : INT_MAX;
              }
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                uint4 w;
                w.x = pack_bf16x2(x[8 * cc + 0], x[8 * cc + 1]);
                w.y = pack_bf16x2(x[8 * cc + 2], x[8 * cc + 3]);
                w.z = pack_bf16x2(x[8 * cc + 4], x[8 * cc + 5]);
                w.w = pack_bf16x2(x[8 * cc + 6], x[8 * cc + 7]);
                const int chunk16 = (4 * h + cc) ^ (lane & 7);
                *reinterpret_cast<uint4*>(buf + lane * 128 + chunk16 * 16) = w;
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int sx = v0 + 64 * jj;
              if (sx < p.c_xlim && row0 < p.c_ylim) tma_store_2d(&p.tmC, buf, sx, row0);
              bulk_commit();
            }
          }
        }
      } else if constexpr (EPI == EPI_TOPK_COLLECT) {
        const bool valid = row < p.rows_valid;
        const float th = valid ? __ldg(p.thr + row) : INFINITY;
        const int v0 = nb * BN;
        int* cv = p.cand_v + static_cast<size_t>(valid ? row : 0) * p.cmax;
        float* cz = p.cand_z + static_cast<size_t>(valid ? row : 0) * p.cmax;
        if (!warp_wait_phase(&tfull[acc], use & 1u, abort_flag, p.status)) break;
        tc_fence_after();
#pragma unroll 1
        for (int j = 0; j < BN / 32; ++j) {
          float x[32];
          __syncwarp();
          tmem_ld32(taddr + 32 * j, x);
          if (j == BN / 32 - 1) release_acc(acc);
          const int cb = v0 + 32 * j;
          uint32_t hits = 0;
#pragma unroll
          for (int t = 0; t < 32; ++t) hits |= (x[t] >= th && cb + t < p.V) ? (1u << t) : 0u;
          while (hits) {
            const int t = __ffs(hits) - 1;
            hits &= hits - 1;
            const int pos = atomicAdd(p.cnt + row, 1);
            if (pos < p.cmax) {
              cv[pos] = cb + t;
              cz[pos] = pick32(x, t);
            }
          }
        }
      } else {
        // EPI_STORE_F32. Two staging buffers per warp, at most one store reading shared memory
        // at a time: box j is staged while store j-1 drains, and store j is issued once store
        // j-1 has read its buffer (which also frees the buffer box j+1 reuses). Stores issued in
        // bursts delay the next unit's operand loads, which share the SM's path to L2; paced,
        // the fp32 output stream of dW costs the main loop less.
        if (!warp_wait_phase(&tfull[acc], use & 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const int y = sp * p.c_split_rows + row0;
#pragma unroll 1
        for (int j = 0; j < BN / 32; ++j, ++ecnt) {
          uint8_t* buf = ebuf0 + (ecnt & 1u) * EPI_BUF_BYTES;
          __syncwarp();  // lane 0 has seen store ecnt-2 read this buffer (before issuing ecnt-1)
          float x[32];
          tmem_ld32(taddr + 32 * j, x);
          if (j == BN / 32 - 1) release_acc(acc);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            const int chunk16 = cc ^ (lane & 7);
            *reinterpret_cast<float4*>(buf + lane * 128 + chunk16 * 16) =
                make_float4(x[4 * cc + 0], x[4 * cc + 1], x[4 * cc + 2], x[4 * cc + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            bulk_wait_read<0>();  // store ecnt-1 has read its buffer
            const int sx = nb * BN + 32 * j;
            if (sx < p.c_xlim && y < p.c_ylim) {
              if (p.c_reduce)
                tma_reduce_add_2d(&p.tmC, buf, sx, y);
              else
                tma_store_2d(&p.tmC, buf, sx, y);
            }
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // the leader's MMAs into this CTA's TMEM are done
  if (warp == 1) {
    tc_fence_after();
    if constexpr (CG == 2)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace fckl
