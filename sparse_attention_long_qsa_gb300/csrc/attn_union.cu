// S5 + S6 for pairs of tokens: one gathered K/V tile serves two tokens, the
// union of their cell lists, with their 2 x 8 query heads in the N = 16
// columns of the MMAs and a per-token mask on every cell.
//
// llama.cpp issue #28734, goodbadwolf's comment on the merged sparse path:
// multi-token batches that do not take the one-column sparse path (a prefill
// ubatch) run a union kernel (ncols1 = 8 tokens x ncols2 = 8 heads) over the
// union of the tokens' selected cells with a mask per token; the same comment
// measures that kernel slower than one column per token for a 5-token verify
// batch.  The per-token kernel (attn.cu) leaves 8 of the 16 N columns of its
// MMAs as zero padding; here they carry a second token's heads, so a cell
// chosen by both tokens of a pair is gathered once.
//
// One thread-block cluster per (token pair (2i, 2i + 1), KV head); every CTA
// first builds the pair's union list on its own (the union is a function of
// the two lists, so no CTA waits for another):
//   - token 0's cells go into an open-addressing hash table in shared memory
//     (cell id -> index in token 0's list);
//   - each cell of token 1 is looked up: a hit marks that entry of token 0's
//     list as token 1's too, a miss keeps the cell for the tail of the union,
//     compacted by a block-wide prefix sum;
//   - union entry i < n0 is token 0's cell i (mask 1, or 3 when token 1 has
//     it), entry n0 + k is token 1's k-th cell outside token 0's list (mask 2).
// The CTAs then take 128-entry tiles of the union (CTA r: tiles r, r + NC, ...)
// as the per-token kernel takes tiles of one list: gather K and V (fp16
// cp.async, or q8_0 through registers and dequantised), S = K Q^T with the
// pair's 16 heads, softmax statistics per column with the column's token mask
// (warps 0-3: token 0's heads, warps 4-7: token 1's, each group reading the
// same TMEM lanes), P for both tokens, O^T = V^T P^T, and a running (max, sum,
// o) per head in registers.  The partials of the 16 (token, head) columns are
// merged over the cluster through distributed shared memory.
//
// Each token gets the attention the per-token kernel computes over its list,
// provided no cell repeats within a token's list (a repeated cell is attended
// once per occurrence by the per-token kernel; here token 1's occurrences of
// a cell that token 0 also lists collapse into one); the tiles hold other
// cells, so the fp16 rounding of P and the order of the sums differ.  Waits
// on the MMA completion barrier are bounded.
#include <atomic>
#include <mutex>

#include "attn_util.cuh"
#include "qsa_internal.cuh"
#include "tc_util.cuh"

namespace qsa {
namespace {

constexpr int kUThreads = 256;
constexpr int kUTile = 128;                 // union entries per MMA tile
constexpr int kUMaxCluster = 16;
constexpr int kUMaxPitch = 4104;            // longest per-token list (top_k 4096, r 8)
constexpr int kUHash = 8192;                // hash slots, a power of two >= 2 x kUMaxPitch
constexpr uint32_t kUTmemCols = 64;         // S: [0,16); O^T half 0: [16,32); half 1: [32,48)

constexpr uint32_t kUOffK = 0;                               // 128 rows x 512 B, 4 atoms of 16 KB
constexpr uint32_t kUOffV = kUOffK + kUTile * 512;           // same layout
constexpr uint32_t kUOffQ = kUOffV + kUTile * 512;           // 16 rows x 512 B: token 0's heads, token 1's
constexpr uint32_t kUOffP = kUOffQ + 16 * 512;               // 16 rows x 256 B
constexpr uint32_t kUOffO = kUOffP + 16 * 256;               // fp32 [NC][16][256/NC] pushed partials
constexpr uint32_t kUOffM = kUOffO + 16 * 256 * 4;           // fp32 [NC][2][16]: per token max[8], sum[8]
constexpr uint32_t kUOffRed = kUOffM + kUMaxCluster * 32 * 4;   // fp32 [2][2][4][8] cross-warp reductions
constexpr uint32_t kUOffCell = kUOffRed + 2 * 64 * 4;        // int [128] the tile's cells
constexpr uint32_t kUOffMask = kUOffCell + kUTile * 4;       // int [128] their token masks
constexpr uint32_t kUOffCell2 = kUOffMask + kUTile * 4;      // int [128] the next tile's cells
constexpr uint32_t kUOffMask2 = kUOffCell2 + kUTile * 4;     // int [128] their masks
constexpr uint32_t kUOffX1 = kUOffMask2 + kUTile * 4;        // int [kUMaxPitch] token 1's extra cells
constexpr uint32_t kUOffHas1 = kUOffX1 + kUMaxPitch * 4;     // u8 [kUMaxPitch] token 0's cells token 1 shares
constexpr uint32_t kUOffScan = (kUOffHas1 + kUMaxPitch + 15u) & ~15u;   // int [8] per-warp counts
constexpr uint32_t kUOffBar = kUOffScan + 32;                // u64 mbarrier
constexpr uint32_t kUOffTmem = kUOffBar + 8;                 // u32 TMEM base address
constexpr uint32_t kUSmem = kUOffTmem + 8 + 1024;            // + alignment slack
static_assert(kUSmem <= 227u * 1024u, "shared memory of the union kernel");
// union-build scratch, dead once the first tile is gathered: token 0's cells
// and the hash table in the K tile, token 1's cells in the V tile
static_assert((kUMaxPitch + kUHash) * 4 <= kUTile * 512, "hash scratch fits in the K tile");
static_assert(kUMaxPitch * 4 <= kUTile * 512, "token 1's cells fit in the V tile");

// kind::f16, fp32 accumulate, fp16 A and B, M = 128, N = 16; A K-major (QK)
// or MN-major (PV), B K-major.
constexpr uint32_t kUIdescQK = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kUIdescPV = kUIdescQK | (1u << 15);

__device__ __forceinline__ uint32_t cell_hash(int c) { return ((uint32_t)c * 2654435761u) >> 19; }   // 13 bits

template <bool kQ8>
__global__ void __launch_bounds__(kUThreads, 1)
k_attn_union(const AttnArgs a, unsigned* err) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_s - raw_s);
  const uint32_t sK = base_s + kUOffK, sV = base_s + kUOffV, sQ = base_s + kUOffQ, sP = base_s + kUOffP;
  float* so = reinterpret_cast<float*>(base + kUOffO);
  float* sml = reinterpret_cast<float*>(base + kUOffM);
  int* scell = reinterpret_cast<int*>(base + kUOffCell);
  int* smask = reinterpret_cast<int*>(base + kUOffMask);
  int* x1 = reinterpret_cast<int*>(base + kUOffX1);
  unsigned char* has1 = base + kUOffHas1;
  int* sscan = reinterpret_cast<int*>(base + kUOffScan);
  const uint32_t bar = base_s + kUOffBar;
  const uint32_t* stmem = reinterpret_cast<const uint32_t*>(base + kUOffTmem);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = warp >> 2;   // the pair's token whose heads this warp group handles
  const int wq = warp & 3;     // the group's quarter of the TMEM lanes (cells, dims)
  float* red = reinterpret_cast<float*>(base + kUOffRed) + grp * 64;
  const int g = blockIdx.y;
  const int t0 = 2 * (int)blockIdx.z, t1 = t0 + 1;
  const bool has_t1 = t1 < a.n_tokens;
  const uint32_t rank = cluster_rank(), NC = cluster_size();
  const int G = a.n_kv_heads, Hq = G * kGqa;
  const int pitch = a.cells_pitch;
  // scores live in the log2 domain: s * attn_scale * log2(e), exponentials by exp2f
  const float scale2 = a.attn_scale * 1.4426950408889634f;

  // ---- prologue (inputs not produced by the preceding index kernels)
  if (warp == 0) tmem_alloc(base_s + kUOffTmem, kUTmemCols);
  if (tid == 0) mbar_init(bar, 1);
  for (int i = tid; i < 16 * 32; i += kUThreads) {
    const int row = i >> 5, c16 = i & 31;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < kGqa || has_t1) {
      const int tok = row < kGqa ? t0 : t1;
      v = __ldg(reinterpret_cast<const uint4*>(a.q + ((int64_t)tok * Hq + g * kGqa + (row & 7)) * kHeadDim +
                                               c16 * 8));
    }
    *reinterpret_cast<uint4*>(base + kUOffQ + sw128(16, row, c16)) = v;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *stmem;

  // ---- the cell lists are written by the index kernels
  grid_dep_wait();
  grid_dep_launch();
  auto clamp_count = [&](int t) {
    const int c = a.count[t];
    return c < 0 ? 0 : (c > pitch ? pitch : c);
  };
  auto checked = [&](int c) {
    if (c < 0 || c >= a.n_cells) {
      atomicOr(err, kErrCell);
      return -1;
    }
    return c;
  };
  const int n0 = clamp_count(t0);
  const int n1 = has_t1 ? clamp_count(t1) : 0;
  const int32_t* row0 = a.cells + (int64_t)t0 * pitch;
  const int32_t* row1 = a.cells + (int64_t)t1 * pitch;

  // ---- the union of the two lists
  int* c0 = reinterpret_cast<int*>(base + kUOffK);
  int* hsh = c0 + kUMaxPitch;
  int* c1 = reinterpret_cast<int*>(base + kUOffV);
  for (int i = tid; i < kUHash; i += kUThreads) hsh[i] = -1;
  for (int i = tid; i < n0; i += kUThreads) {
    c0[i] = checked(row0[i]);
    has1[i] = 0;
  }
  for (int j = tid; j < n1; j += kUThreads) c1[j] = checked(row1[j]);
  __syncthreads();
  for (int i = tid; i < n0; i += kUThreads) {
    const int c = c0[i];
    if (c < 0) continue;
    uint32_t h = cell_hash(c);
    for (int probe = 0; probe < kUHash; ++probe) {   // at most n0 < kUHash slots are taken
      const int prev = atomicCAS(&hsh[h], -1, i);
      if (prev < 0 || c0[prev] == c) break;        // inserted, or the cell is listed already
      h = (h + 1) & (kUHash - 1);
    }
  }
  __syncthreads();
  // token 1's cells: a contiguous run per thread, looked up; shared ones are
  // marked on token 0's entry and dropped, invalid ones dropped (masked
  // either way), the rest counted
  const int per = (n1 + kUThreads - 1) / kUThreads;
  const int j0 = min(n1, tid * per), j1 = min(n1, j0 + per);
  int nx = 0;
  for (int j = j0; j < j1; ++j) {
    const int c = c1[j];
    if (c < 0) continue;
    uint32_t h = cell_hash(c);
    bool found = false;
    for (int probe = 0; probe < kUHash; ++probe) {
      const int v = hsh[h];
      if (v < 0) break;
      if (c0[v] == c) {
        has1[v] = 1;
        found = true;
        break;
      }
      h = (h + 1) & (kUHash - 1);
    }
    if (found) {
      c1[j] = -1;
    } else {
      ++nx;
    }
  }
  int incl = nx;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kWarpAll, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sscan[warp] = incl;
  __syncthreads();
  int at = incl - nx, n1x = 0;
#pragma unroll
  for (int w = 0; w < kUThreads / 32; ++w) {
    const int s = sscan[w];
    if (w < warp) at += s;
    n1x += s;
  }
  for (int j = j0; j < j1; ++j) {
    const int c = c1[j];
    if (c >= 0) x1[at++] = c;
  }
  __syncthreads();   // x1 and has1 complete; the scratch in the K and V tiles is dead
  const int n_union = n0 + n1x;
  const int n_tiles = (n_union + kUTile - 1) / kUTile;

  float run_m[kGqa], run_l[kGqa], acc[2][kGqa];
#pragma unroll
  for (int h = 0; h < kGqa; ++h) {
    run_m[h] = -INFINITY;
    run_l[h] = 0.f;
    acc[0][h] = acc[1][h] = 0.f;
  }
  uint32_t phase = 0;
  bool timed_out = false;
  const int mybit = 1 << grp;

  // fp16: a tile's K and V rows are gathered together (cp.async) at the top
  // of its iteration, the next tile's cells listed meanwhile.  Gathering the
  // next tile's K rows once Q.K^T has completed and its V rows once P.V has
  // (64 KB in flight at a time instead of 128 KB) was measured slower where
  // the rows come from L2 (two tokens sharing most cells: 512-token prefill
  // 361 -> 400 us) and faster where they come from DRAM (523 against 571 us),
  // so the kernel keeps the burst that wins where the union pays.  q8_0: the
  // next tile's int8 rows and scales load into registers under this tile's
  // MMAs and are dequantised into the tiles at the next iteration.  Cell
  // lists alternate between two buffers.
  int* cur = scell;
  int* curm = smask;
  int* nxt = reinterpret_cast<int*>(base + kUOffCell2);
  int* nxtm = reinterpret_cast<int*>(base + kUOffMask2);
  // the cells and masks of union tile `tile` (token 0's ids re-read from its
  // list; an invalid one was flagged above), one entry per thread tid < 128
  auto list_tile = [&](int tile, int* dc, int* dm) {
    const int i = tile * kUTile + tid;
    int c = -1, m = 0;
    if (i < n0) {
      c = row0[i];
      m = 1 | ((int)has1[i] << 1);
    } else if (i < n_union) {
      c = x1[i - n0];
      m = 2;
    }
    if (c < 0 || c >= a.n_cells) {
      c = -1;
      m = 0;
    }
    dc[tid] = c;
    dm[tid] = m;
  };
  const __half* kb = static_cast<const __half*>(a.k_cache);
  const __half* vb = static_cast<const __half*>(a.v_cache);
  auto gather = [&](const int* cells) {
    for (int i = tid; i < kUTile * 32; i += kUThreads) {
      const int row = i >> 5, c16 = i & 31, c = cells[row];
      const int64_t off = ((int64_t)(c < 0 ? 0 : c) * G + g) * kHeadDim + c16 * 8;
      cp_async16(sK + sw128(kUTile, row, c16), kb + off, c >= 0);
      cp_async16(sV + sw128(kUTile, row, c16), vb + off, c >= 0);
    }
  };
  // q8_0: each half warp takes one row at a time, lane l its 16 int8 at dims
  // 16 (l % 16) .. +15 of K and of V and the scale of their q8_0 block (a
  // warp load covers two whole rows); warp w takes rows 16 w + 2 j + l / 16
  const int qc16 = tid & 15, qr0 = 16 * (tid >> 5) + ((tid >> 4) & 1);
  uint4 qk[8], qv[8];
  __half qks[8], qvs[8];    // scales of rows j (not combined in the fetch, so
                            // nothing waits on a load before the MMAs)
  unsigned qvalid = 0u;     // bit j: row qr0 + 2j holds a cell
  auto q8_fetch = [&](const int* cl) {
    qvalid = 0u;
    if (a.n_cells <= 0) return;   // no row to read: every row is stored as zeros
    const int8_t* kq = static_cast<const int8_t*>(a.k_cache);
    const int8_t* vq = static_cast<const int8_t*>(a.v_cache);
    const int64_t nq = a.n_cells * (int64_t)G * kHeadDim;
    const __half* kd = reinterpret_cast<const __half*>(kq + nq);
    const __half* vd = reinterpret_cast<const __half*>(vq + nq);
    // every load is issued (an invalid row reads cell 0's, which exists,
    // and is zeroed when stored), so none waits behind a branch
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = cl[qr0 + 2 * j];
      const int64_t cg = (int64_t)(c < 0 ? 0 : c) * G + g;
      qk[j] = __ldg(reinterpret_cast<const uint4*>(kq + cg * kHeadDim) + qc16);
      qv[j] = __ldg(reinterpret_cast<const uint4*>(vq + cg * kHeadDim) + qc16);
      qks[j] = kd[cg * 8 + (qc16 >> 1)];
      qvs[j] = vd[cg * 8 + (qc16 >> 1)];
      qvalid |= (c >= 0 ? 1u : 0u) << j;
    }
  };
  auto q8_store = [&]() {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const __half2 skf = __half2half2(qks[j]), svf = __half2half2(qvs[j]);
      // lanes 4-7 of each quarter warp store their upper chunk first, so the
      // 8 lanes of a quarter cover the 8 chunk positions of the line
      const int row = qr0 + 2 * j, sw = (qc16 >> 2) & 1, ca = 2 * qc16 + sw, cb = 2 * qc16 + 1 - sw;
      const bool ok = (qvalid >> j) & 1u;
      const uint4 k0 = ok ? dq8(make_uint2(qk[j].x, qk[j].y), skf) : make_uint4(0, 0, 0, 0);
      const uint4 k1 = ok ? dq8(make_uint2(qk[j].z, qk[j].w), skf) : make_uint4(0, 0, 0, 0);
      const uint4 v0 = ok ? dq8(make_uint2(qv[j].x, qv[j].y), svf) : make_uint4(0, 0, 0, 0);
      const uint4 v1 = ok ? dq8(make_uint2(qv[j].z, qv[j].w), svf) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(base + kUOffK + sw128(kUTile, row, ca)) = sw ? k1 : k0;
      *reinterpret_cast<uint4*>(base + kUOffK + sw128(kUTile, row, cb)) = sw ? k0 : k1;
      *reinterpret_cast<uint4*>(base + kUOffV + sw128(kUTile, row, ca)) = sw ? v1 : v0;
      *reinterpret_cast<uint4*>(base + kUOffV + sw128(kUTile, row, cb)) = sw ? v0 : v1;
    }
  };

  if ((int)rank < n_tiles) {
    if (tid < kUTile) list_tile((int)rank, cur, curm);
    __syncthreads();
    if constexpr (kQ8) q8_fetch(cur);
  }
  for (int tile = (int)rank; tile < n_tiles; tile += (int)NC) {
    const bool has_next = tile + (int)NC < n_tiles;
    if constexpr (kQ8) {
      q8_store();
    } else {
      gather(cur);
    }
    if (has_next && tid < kUTile) list_tile(tile + (int)NC, nxt, nxtm);
    if constexpr (!kQ8) asm volatile("cp.async.wait_all;\n" ::: "memory");
    fence_async_smem();
    tc_fence_before();
    __syncthreads();   // K and V tiles complete; the next tile's cells listed
    tc_fence_after();
    if constexpr (kQ8) {
      if (has_next) q8_fetch(nxt);
    }

    // 2. S[cell][col] = K . Q^T for the pair's 16 heads
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const uint64_t ad = smem_desc(sK + (kk >> 2) * (kUTile * 128) + (kk & 3) * 32, 16, 1024);
        const uint64_t bd = smem_desc(sQ + (kk >> 2) * (16 * 128) + (kk & 3) * 32, 16, 1024);
        mma_f16(tmem, ad, bd, kUIdescQK, kk > 0);
      }
      mma_commit(bar);
    }
    if (!mbar_wait(bar, phase)) timed_out = true;
    phase ^= 1;
    tc_fence_after();

    // 3. per group: its token's columns, masked by its bit; statistics by
    // warp reduce-scatter (lanes 4k hold head k's), P rows 8 grp + h
    float sv[kGqa], tmax[kGqa], pe[kGqa];
    tmem_ld8(tmem + ((uint32_t)(32 * wq) << 16) + 8 * grp, sv);
    const int cell = 32 * wq + lane;
    const bool valid = (curm[cell] & mybit) != 0;
#pragma unroll
    for (int h = 0; h < kGqa; ++h) sv[h] = valid ? sv[h] * scale2 : -INFINITY;
    {
      const float m = warp_reduce8(sv, lane, OpMax());
      if ((lane & 3) == 0) red[wq * 8 + (lane >> 2)] = m;
    }
    bar_half(1 + grp);
#pragma unroll
    for (int h = 0; h < kGqa; ++h) tmax[h] = fmaxf(fmaxf(red[h], red[8 + h]), fmaxf(red[16 + h], red[24 + h]));
#pragma unroll
    for (int h = 0; h < kGqa; ++h) {
      const float p = (tmax[h] == -INFINITY) ? 0.f : exp2f(sv[h] - tmax[h]);
      const __half ph = __float2half_rn(p);
      pe[h] = __half2float(ph);   // the sum uses the rounded p the MMA sees
      const int prow = 8 * grp + h;
      const uint32_t off = (uint32_t)(cell >> 6) * (16 * 128) + prow * 128 +
                           ((((uint32_t)(cell & 63) >> 3) ^ (uint32_t)(prow & 7)) << 4) + (cell & 7) * 2;
      *reinterpret_cast<__half*>(base + kUOffP + off) = ph;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();   // both tokens' P rows written
    tc_fence_after();

    // 4. O^T[dim][col] = V^T . P^T, two halves of 128 dims; row sums reduced
    // while the MMAs run
    if (tid == 0) {
#pragma unroll
      for (int mh = 0; mh < 2; ++mh) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = smem_desc(sV + mh * 2 * (kUTile * 128) + kk * 2048, kUTile * 128, 1024);
          const uint64_t bd = smem_desc(sP + (kk >> 2) * (16 * 128) + (kk & 3) * 32, 16, 1024);
          mma_f16(tmem + 16 + 16 * mh, ad, bd, kUIdescPV, kk > 0);
        }
      }
      mma_commit(bar);
    }
    {
      const float e = warp_reduce8(pe, lane, OpAdd());
      if ((lane & 3) == 0) red[32 + wq * 8 + (lane >> 2)] = e;
    }
    bar_half(1 + grp);
    float tsum[kGqa];
#pragma unroll
    for (int h = 0; h < kGqa; ++h) tsum[h] = (red[32 + h] + red[40 + h]) + (red[48 + h] + red[56 + h]);
    if (!mbar_wait(bar, phase)) timed_out = true;
    phase ^= 1;
    tc_fence_after();

    // 5. merge the tile into the running state (dims 32 wq + lane and + 128)
    float o0[8], o1[8];
    tmem_ld8(tmem + ((uint32_t)(32 * wq) << 16) + 16 + 8 * grp, o0);
    tmem_ld8(tmem + ((uint32_t)(32 * wq) << 16) + 32 + 8 * grp, o1);
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
    tc_fence_before();
    __syncthreads();   // tiles, P and tensor memory free for the next tile
    tc_fence_after();
    int* t_ = cur;
    cur = nxt;
    nxt = t_;
    t_ = curm;
    curm = nxtm;
    nxtm = t_;
  }
  if (timed_out) atomicOr(err, kErrTimeout);

  // ---- push the 16 columns' partials to the CTAs owning each dim range,
  // then every CTA reduces its range from its own shared memory
  const int dpc = (kHeadDim + (int)NC - 1) / (int)NC;   // dims per owner (a multiple of 4)
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int d = half * 128 + 32 * wq + lane;
    const uint32_t owner = (uint32_t)(d / dpc), e = (uint32_t)(d % dpc);
#pragma unroll
    for (int h = 0; h < kGqa; ++h)
      st_dsmem_f32(dsmem_addr(&so[((int)rank * 16 + 8 * grp + h) * dpc + e], owner), acc[half][h]);
  }
  if ((tid & 127) < (int)NC) {
    const uint32_t dst = dsmem_addr(&sml[(int)rank * 32 + 16 * grp], (uint32_t)(tid & 127));
    st_dsmem_f32x4(dst, make_float4(run_m[0], run_m[1], run_m[2], run_m[3]));
    st_dsmem_f32x4(dst + 16, make_float4(run_m[4], run_m[5], run_m[6], run_m[7]));
    st_dsmem_f32x4(dst + 32, make_float4(run_l[0], run_l[1], run_l[2], run_l[3]));
    st_dsmem_f32x4(dst + 48, make_float4(run_l[4], run_l[5], run_l[6], run_l[7]));
  }
  cluster_sync();   // all pushes have landed; nobody touches a peer after this
  {
    // normalised weight of each (partial p, column): a column's partials in
    // 16 consecutive lanes; then one output per thread
    float* wgt = reinterpret_cast<float*>(base + kUOffQ);   // the Q tile is no longer read
    const int col = tid >> 4, p = tid & 15, gr = col >> 3, h = col & 7;
    const float mp = p < (int)NC ? sml[p * 32 + 16 * gr + h] : -INFINITY;
    const float lp = p < (int)NC ? sml[p * 32 + 16 * gr + 8 + h] : 0.f;
    float mx = mp;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kWarpAll, mx, o));
    const float w = (mp == -INFINITY) ? 0.f : exp2f(mp - mx);
    float den = w * lp;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) den += __shfl_xor_sync(kWarpAll, den, o);
    wgt[p * 16 + col] = den > 0.f ? w / den : 0.f;
    __syncthreads();
    const int d0 = (int)rank * dpc;
    for (int i = tid; i < 16 * dpc; i += kUThreads) {
      const int c = i / dpc, e = i % dpc, d = d0 + e;
      if (d >= kHeadDim || (c >= kGqa && !has_t1)) continue;
      float o = 0.f;
      for (int q = 0; q < (int)NC; ++q) o = fmaf(wgt[q * 16 + c], so[(q * 16 + c) * dpc + e], o);
      const int tok = c < kGqa ? t0 : t1;
      a.out[((int64_t)tok * Hq + g * kGqa + (c & 7)) * kHeadDim + d] = o;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kUTmemCols);
}

constexpr int kUMaxDevices = 64;

// Cluster size for `clusters` clusters of up to `tiles` tiles each, as the
// per-token kernel chooses it: the largest size (<= 16, <= tiles) whose
// clusters all fit at once, else the fewest waves x (1 + tiles per CTA).
template <bool kQ8>
cudaError_t pick_union_cluster(int64_t clusters, int tiles, int* nc_out) {
  static int max_active[kUMaxDevices][5];
  static std::atomic<bool> configured[kUMaxDevices];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kUMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(k_attn_union<kQ8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kUSmem);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(k_attn_union<kQ8>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      for (int i = 0; i < 5; ++i) {
        const int nc = 16 >> i;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)nc, 1, 1);
        cfg.blockDim = dim3(kUThreads, 1, 1);
        cfg.dynamicSmemBytes = (size_t)kUSmem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = (unsigned)nc;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_attn_union<kQ8>, &cfg) != cudaSuccess) {
          (void)cudaGetLastError();
          n = 0;
        }
        max_active[dev][i] = n;
      }
      configured[dev].store(true, std::memory_order_release);
    }
  }
  const int want = tiles < kUMaxCluster ? (tiles > 0 ? tiles : 1) : kUMaxCluster;
  int nc = 0;
  for (int i = 0; i < 5; ++i) {
    const int c = 16 >> i;
    if (c > want || max_active[dev][i] <= 0) continue;
    if (clusters <= max_active[dev][i]) {
      nc = c;
      break;
    }
  }
  if (nc == 0) {
    int64_t best = -1;
    for (int i = 0; i < 5; ++i) {
      const int c = 16 >> i;
      if (c > want || max_active[dev][i] <= 0) continue;
      const int64_t waves = ceil_div(clusters, (int64_t)max_active[dev][i]);
      const int64_t cost = waves * (1 + ceil_div((int64_t)tiles, (int64_t)c));
      if (best < 0 || cost < best) {
        best = cost;
        nc = c;
      }
    }
    if (nc == 0) nc = 1;
  }
  *nc_out = nc;
  return cudaSuccess;
}

template <bool kQ8>
cudaError_t launch_union(const AttnArgs& a, unsigned* err, cudaStream_t stream) {
  const int64_t pairs = ceil_div(a.n_tokens, 2);
  const int64_t clusters = pairs * a.n_kv_heads;
  // the union of two lists: at most two lists' tiles
  const int tiles = (int)ceil_div(2 * (int64_t)a.cells_pitch, kUTile);
  int nc = 1;
  cudaError_t e = pick_union_cluster<kQ8>(clusters, tiles, &nc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nc, (unsigned)a.n_kv_heads, (unsigned)pairs);
  cfg.blockDim = dim3(kUThreads, 1, 1);
  cfg.dynamicSmemBytes = kUSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_attn_union<kQ8>, a, err);
}

}  // namespace

int union_attn_max_pitch() { return kUMaxPitch; }

cudaError_t launch_sparse_attn_union(const AttnArgs& a, unsigned* err, cudaStream_t stream) {
  if (a.n_tokens <= 0) return cudaSuccess;
  if (a.cells_pitch > kUMaxPitch) return cudaErrorInvalidValue;
  prof_before(kKAttn, stream);
  cudaError_t e = a.kv_q8 ? launch_union<true>(a, err, stream) : launch_union<false>(a, err, stream);
  prof_after(kKAttn, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qsa
