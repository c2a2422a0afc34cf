// S5 + S6 for calls with many tokens (the prefill ubatch), fp16 K/V: the
// same attention as k_attn_tc (llama.cpp issue #28734, fix summary, lever1:
// attention over only the selected K/V set; sparse256: DKQ = DV = 256, 8
// query heads per KV head), laid out so that two CTAs share an SM.
//
// A gather of 512-byte rows reaches about 4.8 TB/s when one CTA per SM
// issues it and about 6.2 TB/s with two, so this variant keeps each CTA
// under half an SM: tiles of 64 cells (32 KB of K or of V per stage, three
// stages), at most 128 registers per thread, ~108 KB of shared memory.  Each
// (token, KV head) is one cluster of two CTAs; CTA r takes tiles r, r + 2, ...
// of the token's cell list.  Per CTA, warps 4-7 gather (load 2i: tile i's K
// rows, load 2i + 1: its V rows, over three rotating stages; full and empty
// mbarriers, every wait bounded) and warps 0-3 run, per tile:
//   S = K . Q^T   M = 128, N = 16, K = 256 (16 tcgen05.mma); rows 64-127 of
//                 the M = 128 operand are the next 8 KB of shared memory (the
//                 next column block, stage or the Q tile) and are masked;
//   softmax       one cell per thread of warps 0-1 (TMEM lanes 0-63), the
//                 tile's statistics by warp reduce-scatter, P (fp16) to
//                 shared memory;
//   O^T = V^T P^T M = 128 dims (two halves), N = 16, K = 64 cells (8 MMAs);
//   merge         into a running (max, sum, o) in registers.
// After both CTAs' loops the cluster synchronises, CTA 1 stores its
// partial into CTA 0's first stage (distributed shared memory), the
// cluster synchronises again and CTA 0 merges the two and writes the output.
#include <atomic>
#include <mutex>

#include "attn_pf.cuh"
#include "attn_util.cuh"
#include "qsa_internal.cuh"
#include "tc_util.cuh"

namespace qsa {
namespace {

constexpr int kPfThreads = 256;
constexpr int kPfTile = 64;                                // cells per tile
constexpr int kPfNC = 2;                                   // CTAs per (token, KV head)
constexpr int kPfStages = 3;
constexpr uint32_t kPfStageBytes = kPfTile * 512u;         // 64 rows x 256 fp16, 4 column blocks of 8 KB
// shared-memory layout (offsets from a 1024-byte aligned base); the Q tile
// follows the last stage, so the M = 128 reads past a stage's last column
// block stay inside the CTA's shared memory
constexpr uint32_t kPfOffQ = kPfStages * kPfStageBytes;    // 16 rows x 512 B
constexpr uint32_t kPfOffP = kPfOffQ + 16 * 512;           // 16 rows x 128 B (64 cells)
constexpr uint32_t kPfOffRed = kPfOffP + 16 * 128;         // fp32 [2][4][8] cross-warp reductions
constexpr uint32_t kPfOffCell = kPfOffRed + 256;           // int [3][64] the stages' tiles' cells
constexpr uint32_t kPfOffBar = kPfOffCell + kPfStages * kPfTile * 4;   // u64 full[3], empty[3], mma
constexpr uint32_t kPfOffTmem = kPfOffBar + 8 * (2 * kPfStages + 1);
constexpr uint32_t kPfSmem = kPfOffTmem + 16 + 1024;       // + alignment slack
constexpr uint32_t kPfTmemCols = 64;                       // S: [0,16); O halves: [16,32), [32,48)
static_assert(2 * (kPfSmem + 1024) <= 228u * 1024u, "two CTAs per SM");
static_assert(16 * 512 >= (128 - kPfTile) * 128, "the M = 128 read past the last stage stays in the Q tile");
// the peer's partial in stage 0 after the loops: fp32 o[8][256], m[8], l[8]
static_assert(8 * 256 * 4 + 64 <= kPfStageBytes, "partial fits in a stage");

// kind::f16: fp32 accumulate, fp16 A and B, M = 128, N = 16; A K-major (QK)
// or MN-major (PV), B K-major
constexpr uint32_t kPfIdescQK = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kPfIdescPV = kPfIdescQK | (1u << 15);

__device__ __forceinline__ void pf_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

__global__ void __launch_bounds__(kPfThreads, 2) k_attn_pf(const AttnArgs a, unsigned* err) {
  extern __shared__ unsigned char pf_smem_raw[];
  const uint32_t raw_s = smem_u32(pf_smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  unsigned char* base = pf_smem_raw + (base_s - raw_s);
  const uint32_t sQ = base_s + kPfOffQ, sP = base_s + kPfOffP;
  float* sred = reinterpret_cast<float*>(base + kPfOffRed);
  int* scl = reinterpret_cast<int*>(base + kPfOffCell);
  const uint32_t bfull = base_s + kPfOffBar, bempty = bfull + 8 * kPfStages, bmma = bempty + 8 * kPfStages;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y, t = blockIdx.z;
  const uint32_t rank = cluster_rank(), NC = cluster_size();
  const int G = a.n_kv_heads, Hq = G * kGqa;
  const float scale2 = a.attn_scale * 1.4426950408889634f;   // scores in the log2 domain

  // ---- prologue (inputs only): tensor memory, barriers, the Q tile, P rows 8-15
  if (warp == 0) tmem_alloc(base_s + kPfOffTmem, kPfTmemCols);
  if (tid == 0) {
    for (int q = 0; q < kPfStages; ++q) {
      mbar_init(bfull + 8 * q, 128);
      mbar_init(bempty + 8 * q, 1);
    }
    mbar_init(bmma, 1);
  }
  {
    const __half* qg = a.q + ((int64_t)t * Hq + g * kGqa) * kHeadDim;
    for (int i = tid; i < 16 * 32; i += kPfThreads) {
      const int row = i >> 5, c16 = i & 31;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row < kGqa) v = __ldg(reinterpret_cast<const uint4*>(qg + row * kHeadDim + c16 * 8));
      *reinterpret_cast<uint4*>(base + kPfOffQ + sw128(16, row, c16)) = v;
    }
    for (int i = tid; i < 8 * 8; i += kPfThreads) {
      const int row = 8 + (i >> 3), c16 = i & 7;
      *reinterpret_cast<uint4*>(base + kPfOffP + sw128(16, row, c16)) = make_uint4(0, 0, 0, 0);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<const uint32_t*>(base + kPfOffTmem);

  // ---- the cell list and count are written by the index kernels
  grid_dep_wait();
  grid_dep_launch();
  const int32_t* crow = a.cells + (int64_t)t * a.cells_pitch;
  int cnt = a.count[t];
  cnt = cnt < 0 ? 0 : (cnt > a.cells_pitch ? a.cells_pitch : cnt);
  const int n_tiles = (cnt + kPfTile - 1) / kPfTile;
  const int n_my = n_tiles > (int)rank ? (n_tiles - (int)rank + (int)NC - 1) / (int)NC : 0;

  float run_m[kGqa], run_l[kGqa], acc[2][kGqa];
#pragma unroll
  for (int h = 0; h < kGqa; ++h) {
    run_m[h] = -INFINITY;
    run_l[h] = 0.f;
    acc[0][h] = acc[1][h] = 0.f;
  }
  bool timed_out = false;

  if (warp >= 4) {
    // ---- gather warps: load L = 2i (tile i's K) or 2i + 1 (its V) into stage L % 3
    const int tx = tid - 128;
    const __half* kb = static_cast<const __half*>(a.k_cache);
    const __half* vb = static_cast<const __half*>(a.v_cache);
    for (int L = 0; L < 2 * n_my; ++L) {
      const int st = L % kPfStages, use = L / kPfStages, i = L >> 1;
      if (!mbar_wait(bempty + 8 * st, (uint32_t)((use & 1) ^ 1))) timed_out = true;
      int* cells = scl + (i % kPfStages) * kPfTile;
      if ((L & 1) == 0) {
        const int c0 = ((int)rank + i * (int)NC) * kPfTile, nvt = min(kPfTile, cnt - c0);
        if (tx < kPfTile) {
          int c = -1;
          if (tx < nvt) {
            c = crow[c0 + tx];
            if (c < 0 || c >= a.n_cells) {
              atomicOr(err, kErrCell);
              c = -1;
            }
          }
          cells[tx] = c;
        }
        bar_half(2);   // every row's cell is listed before any copy reads it
      }
      const __half* src = (L & 1) ? vb : kb;
      const uint32_t dst = base_s + st * kPfStageBytes;
      for (int k = tx; k < kPfTile * 32; k += 128) {
        const int row = k >> 5, c16 = k & 31, c = cells[row];
        const int64_t off = ((int64_t)(c < 0 ? 0 : c) * G + g) * kHeadDim + c16 * 8;
        cp_async16(dst + sw128(kPfTile, row, c16), src + off, c >= 0);
      }
      asm volatile("cp.async.commit_group;\n" ::: "memory");
      if (L > 0) {
        asm volatile("cp.async.wait_group 1;\n" ::: "memory");   // load L - 1 has landed
        fence_async_smem();
        pf_arrive(bfull + 8 * ((L - 1) % kPfStages));
      }
    }
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    fence_async_smem();
    if (n_my > 0) pf_arrive(bfull + 8 * ((2 * n_my - 1) % kPfStages));
  } else {
    // ---- warps 0-3: the tiles' MMAs, softmax and merge
    uint32_t phase = 0;
    for (int i = 0; i < n_my; ++i) {
      const int tile = (int)rank + i * (int)NC;
      const int nv = min(kPfTile, cnt - tile * kPfTile);
      const int sk = (2 * i) % kPfStages, sv = (2 * i + 1) % kPfStages;
      const uint32_t uK = base_s + sk * kPfStageBytes, uV = base_s + sv * kPfStageBytes;
      const int* cells = scl + (i % kPfStages) * kPfTile;
      if (!mbar_wait(bfull + 8 * sk, (uint32_t)(((2 * i) / kPfStages) & 1))) timed_out = true;
      tc_fence_after();
      // S[cell][head] = K . Q^T
      if (tid == 0) {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint64_t ad = smem_desc(uK + (kk >> 2) * (kPfTile * 128) + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc(sQ + (kk >> 2) * (16 * 128) + (kk & 3) * 32, 16, 1024);
          mma_f16(tmem, ad, bd, kPfIdescQK, kk > 0);
        }
        mma_commit(bmma);
      }
      if (!mbar_wait(bmma, phase)) timed_out = true;
      phase ^= 1;
      tc_fence_after();
      if (tid == 0) pf_arrive(bempty + 8 * sk);   // Q.K^T has completed: the K stage is free
      // tile softmax statistics and P, one cell per thread (cells >= 64 are
      // the masked rows of the M = 128 product)
      float sv8[kGqa], tmax[kGqa], pe[kGqa];
      tmem_ld8(tmem + ((uint32_t)(32 * warp) << 16), sv8);
      const int cell = 32 * warp + lane;
      const bool valid = cell < nv && cells[cell] >= 0;
#pragma unroll
      for (int h = 0; h < kGqa; ++h) sv8[h] = valid ? sv8[h] * scale2 : -INFINITY;
      {
        const float m = warp_reduce8(sv8, lane, OpMax());
        if ((lane & 3) == 0) sred[warp * 8 + (lane >> 2)] = m;
      }
      bar_half(1);
#pragma unroll
      for (int h = 0; h < kGqa; ++h) tmax[h] = fmaxf(fmaxf(sred[h], sred[8 + h]), fmaxf(sred[16 + h], sred[24 + h]));
#pragma unroll
      for (int h = 0; h < kGqa; ++h) {
        const float p = (tmax[h] == -INFINITY) ? 0.f : exp2f(sv8[h] - tmax[h]);
        const __half ph = __float2half_rn(p);
        pe[h] = __half2float(ph);   // the sum uses the rounded p the MMA sees
        if (cell < kPfTile) {
          // P row h, column `cell`: chunk cell / 8 of the 128-byte row, element cell % 8
          const uint32_t off = h * 128 + ((((uint32_t)cell >> 3) ^ (uint32_t)(h & 7)) << 4) + (cell & 7) * 2;
          *reinterpret_cast<__half*>(base + kPfOffP + off) = ph;
        }
      }
      fence_async_smem();
      tc_fence_before();
      bar_half(1);
      tc_fence_after();
      if (!mbar_wait(bfull + 8 * sv, (uint32_t)(((2 * i + 1) / kPfStages) & 1))) timed_out = true;
      tc_fence_after();
      // O^T[dim][head] = V^T . P^T, two halves of 128 dims; the tile's row
      // sums are reduced while the MMAs run
      if (tid == 0) {
#pragma unroll
        for (int mh = 0; mh < 2; ++mh) {
#pragma unroll
          for (int kk = 0; kk < kPfTile / 16; ++kk) {
            const uint64_t ad = smem_desc(uV + mh * 2 * (kPfTile * 128) + kk * 2048, kPfTile * 128, 1024);
            const uint64_t bd = smem_desc(sP + kk * 32, 16, 1024);
            mma_f16(tmem + 16 + 16 * mh, ad, bd, kPfIdescPV, kk > 0);
          }
        }
        mma_commit(bmma);
      }
      {
        const float e = warp_reduce8(pe, lane, OpAdd());
        if ((lane & 3) == 0) sred[32 + warp * 8 + (lane >> 2)] = e;
      }
      bar_half(1);
      float tsum[kGqa];
#pragma unroll
      for (int h = 0; h < kGqa; ++h) tsum[h] = (sred[32 + h] + sred[40 + h]) + (sred[48 + h] + sred[56 + h]);
      if (!mbar_wait(bmma, phase)) timed_out = true;
      phase ^= 1;
      tc_fence_after();
      if (tid == 0) pf_arrive(bempty + 8 * sv);   // P.V has completed: the V stage is free
      // merge the tile into the running state (dims 32 warp + lane and +128)
      float o0[kGqa], o1[kGqa];
      tmem_ld8(tmem + ((uint32_t)(32 * warp) << 16) + 16, o0);
      tmem_ld8(tmem + ((uint32_t)(32 * warp) << 16) + 32, o1);
#pragma unroll
      for (int h = 0; h < kGqa; ++h) {
        const float mn = fmaxf(run_m[h], tmax[h]);
        const float fa = (run_m[h] == -INFINITY) ? 0.f : exp2f(run_m[h] - mn);
        const float fb = (tmax[h] == -INFINITY) ? 0.f : exp2f(tmax[h] - mn);
        acc[0][h] = acc[0][h] * fa + o0[h] * fb;
        acc[1][h] = acc[1][h] * fa + o1[h] * fb;
        run_l[h] = run_l[h] * fa + tsum[h] * fb;
        run_m[h] = mn;
      }
    }
  }
  if (timed_out) atomicOr(err, kErrTimeout);

  // ---- the two CTAs' partials: CTA 1 stores its (o, m, l) into CTA 0's
  // stage 0 once both loops are done; CTA 0 merges and writes the output
  tc_fence_before();
  __syncthreads();
  float* peer = reinterpret_cast<float*>(base);   // o[8][256], then m[8], l[8]
  if (NC > 1) {
    cluster_sync();   // both CTAs are done with their stages
    if (rank == 1 && warp < 4) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int d = half * 128 + 32 * warp + lane;
#pragma unroll
        for (int h = 0; h < kGqa; ++h) st_dsmem_f32(dsmem_addr(&peer[h * kHeadDim + d], 0), acc[half][h]);
      }
      if (tid < kGqa) {
        float m = 0.f, l = 0.f;   // head tid's statistics (no dynamic register index)
#pragma unroll
        for (int h = 0; h < kGqa; ++h)
          if (h == tid) {
            m = run_m[h];
            l = run_l[h];
          }
        st_dsmem_f32(dsmem_addr(&peer[kGqa * kHeadDim + tid], 0), m);
        st_dsmem_f32(dsmem_addr(&peer[kGqa * kHeadDim + kGqa + tid], 0), l);
      }
    }
    cluster_sync();   // the partial has landed; nobody touches a peer after this
  }
  if (rank == 0 && warp < 4) {
#pragma unroll
    for (int h = 0; h < kGqa; ++h) {
      float o0 = acc[0][h], o1 = acc[1][h], l = run_l[h];
      if (NC > 1) {
        const float mp = peer[kGqa * kHeadDim + h], lp = peer[kGqa * kHeadDim + kGqa + h];
        const float mn = fmaxf(run_m[h], mp);
        const float fa = (run_m[h] == -INFINITY) ? 0.f : exp2f(run_m[h] - mn);
        const float fb = (mp == -INFINITY) ? 0.f : exp2f(mp - mn);
        o0 = o0 * fa + peer[h * kHeadDim + 32 * warp + lane] * fb;
        o1 = o1 * fa + peer[h * kHeadDim + 128 + 32 * warp + lane] * fb;
        l = l * fa + lp * fb;
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float* orow = a.out + ((int64_t)t * Hq + g * kGqa + h) * kHeadDim;
      orow[32 * warp + lane] = o0 * inv;
      orow[128 + 32 * warp + lane] = o1 * inv;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kPfTmemCols);
}

constexpr int kPfMaxDevices = 64;

}  // namespace

bool attn_pf_eligible(const AttnArgs& a) { return !a.kv_q8 && a.cells_pitch >= 4 * kPfTile; }

cudaError_t launch_attn_pf(const AttnArgs& a, unsigned* err, cudaStream_t stream) {
  static std::atomic<bool> configured[kPfMaxDevices];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kPfMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(k_attn_pf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPfSmem);
      if (e != cudaSuccess) return e;
      configured[dev].store(true, std::memory_order_release);
    }
  }
  return launch_pdl(k_attn_pf, dim3((unsigned)kPfNC, (unsigned)a.n_kv_heads, (unsigned)a.n_tokens),
                    dim3(kPfThreads), kPfSmem, stream, (unsigned)kPfNC, a, err);
}

}  // namespace qsa
