// attn_dense.cu -- dense-causal partial MLA attention (output + LSE, no sink)
// for context-parallel prefill, bf16 latent KV, on sm_103a.
//
// "[DeepSeekV4][PCP] Enable context-parallel prefill for hybrid KV and
// MegaMoE", "Implementation summary": per-shard partial attention merged
// later by LSE; "[Core] Add MRV2 virtual-batch PCP for MLA", "DualChunkSwap
// partitioning": each shard's rows attend causally over the full latent KV.
//
// One CTA = 64 query rows (G tokens x Hc heads of consecutive shard rows).
//   * Score GEMM key-major: S^T = K . Q^T, M = 128 keys, N = 64 rows, K = 576,
//     into one of two TMEM buffers, so the score GEMM of tile j+1 runs while
//     the softmax of tile j does.  PV GEMM: O^T += V^T . P^T, M = 128 dv x 4
//     chunks, N = 64, K = 128 keys; O^T stays in TMEM (256 columns).
//   * One ring of four 32 KB slots streams everything the tensor core reads:
//     K of a tile as five slots (k-block pairs of [128 keys x 64 dims], the
//     rope k-block alone) and V of a tile as four 128-dv chunks [128 keys x
//     128 dv] -- a second read of the same L2-resident rows, so neither GEMM
//     holds shared memory the other needs.  The sequence interleaves the two
//     GEMMs item by item (V(t) chunk c, then K(t+2) pair c): with blocks of
//     one GEMM's items, each issuer waited for the other's slots to turn over.  Two producer threads fill it with TMA (128-byte swizzle),
//     item n from warp 2 + n % 2: a single issuing thread caps the TMA
//     ingress of an SM near 40 B/clk, two reach about twice that.
//   * Two threads issue the tcgen05.mma: warp 0 the score GEMMs, warp 1 the
//     PV GEMMs, each taking its own items of the ring sequence.  One thread issues an MMA only
//     every ~80 cycles, while the tensor core finishes an N = 64 MMA in
//     ~48 (its shared-memory operand reads), so one issuer would leave it
//     idle.  Warps 4-11 are two softmax warpgroups of 32 rows each (thread
//     i = TMEM lane i = key i of a tile / dv i of an O^T chunk).
//   * Tiles that lie inside every row's causal range skip the mask.
//   * Every wait is bounded; on expiry the CTA records CPMLA_ERR_TIMEOUT,
//     drains its copies and MMAs, and exits.
#include <cmath>

#include "attn_common.cuh"

namespace cpmla {
namespace {

constexpr int kR = 64;                      // query rows per CTA (MMA N)
constexpr int kRW = 32;                     // rows per softmax warpgroup
constexpr int kNS = 4;                      // ring slots
constexpr int kProducers = 2;               // TMA-issuing threads (warps 2-3)
constexpr int kSlotBytes = 2 * kKbBytes;    // 32 KB: two k-blocks or one 128-dv chunk
constexpr int kKPairs = 5;                  // K of a tile: k-block pairs 0-3 + rope
constexpr int kVChunks = 4;                 // V of a tile: 128-dv chunks
constexpr int kPBytes = kTileKeys * kR * 2; // P^T, 16 KB
constexpr int kFullBars = 4 * kNS;          // ring item n lands on full[n % kFullBars]
constexpr uint32_t kTmemCols = 512;         // S^T x2 (128) + O^T (256)

struct DenseCtrl {
  // Ring item n lands on full[n % kFullBars]: four barriers per slot, used
  // by successive items of the slot in turn.  The two MMA issuers each wait
  // only for their own items, so one of them can wait for item n while an
  // earlier item of the same slot (the other's) has not landed; with too few
  // barriers per slot the parity test would then pass a phase early.  With
  // four, the item that last used the barrier (n - 4 kNS) has always landed
  // by then -- checked against a randomised event model of this ring order.
  uint64_t full[kFullBars];
  uint64_t empty[kNS];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t p_free;
  uint64_t o_full;
  uint64_t drain[2];
  uint64_t q_full;  // Q rows landed (TMA path)
  uint32_t tmem_base;
  int abort;
  int n_tiles;
  int open_lo, open_hi;  // tiles j in [open_lo, open_hi) need no mask
  int bflag[2][2];
  int need_rescale[2];
  int64_t tile_lo;  // global KV row of key 0 of tile 0
  int rlo[kR];      // per row: valid keys relative to tile_lo, inclusive
  int rhi[kR];
  float red[2][4][32];
  float m_ref[kR];
  float alpha[kR];
  float lse[kR];
  alignas(16) float inv_l[kR];
  alignas(16) float sfac[kR];  // merged output: sink factor per row
  int64_t obase[kR];  // partial output: element offset of a row in o_part, -1: none
  int gtok[kR];    // merged output: global token a row writes, or -1
  int64_t tlo[kR], thi[kR];  // per token of the item: valid keys (global rows, inclusive)
  int ttok[kR];              // per token: global token, -1 past the last shard row
  int town[kR];              // merged, per token: the token if its row owns it, else -1
};

constexpr int kQBytes = kR * CPMLA_DQK * 2;
constexpr int kSmem = 1024 + kQBytes + kPBytes + kNS * kSlotBytes + (int)sizeof(DenseCtrl);
static_assert(kSmem <= 232448, "shared memory budget");

// Bounded wait that ignores the abort flag (used to drain own copies).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity) && global_timer_ns() - t0 < kWaitLimitNs) {
  }
}

// Valid key range of shard row i, as global KV rows (inclusive), or lo > hi.
__device__ __forceinline__ void row_range(const AttnArgs &a, int i, int64_t &lo, int64_t &hi) {
  const int64_t base = a.kv_start[a.req[i]];
  lo = 0;
  hi = a.pos[i];
  if (a.kv_lo) lo = lo > a.kv_lo[i] ? lo : a.kv_lo[i];
  if (a.kv_hi) hi = hi < a.kv_hi[i] ? hi : a.kv_hi[i];
  lo += base;
  hi += base;
  if (hi > a.s_kv - 1) hi = a.s_kv - 1;
  if (lo < 0) lo = 0;
}

// Ring order: K(0), K(1), then block t = 0, 1, ...: V(t) chunk c followed by
// K(t+2) pair c (c = 0..3), then the rope of K(t+2); a block with no K(t+2)
// (t >= n - 2) holds V(t) alone.  Interleaving the two GEMMs' items lets their
// issuers run side by side instead of taking turns over the four slots.
__device__ __forceinline__ uint32_t ring_block_base(int t, int n) {
  const int nk = n < 2 ? n : 2;            // K(0), K(1)
  const int nfull = n > 2 ? n - 2 : 0;     // blocks with a K part
  const int tf = t < nfull ? t : nfull;
  return (uint32_t)(5 * nk + 9 * tf + 4 * (t - tf));
}
__device__ __forceinline__ uint32_t ring_pos_k(int i, int p) {  // i < n
  return i < 2 ? (uint32_t)(5 * i + p) : (uint32_t)(10 + 9 * (i - 2) + (p < 4 ? 2 * p + 1 : 8));
}
__device__ __forceinline__ uint32_t ring_pos_v(int j, int ch, int n) {
  return ring_block_base(j, n) + (uint32_t)(j + 2 < n ? 2 * ch : ch);
}

// MERGED: the epilogue writes each owned token's merged result
// (AttnArgs::o_out) instead of the partial (o_part / lse_part).
template <bool MERGED>
__global__ void __launch_bounds__(kThreads, 1)
    mla_dense_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap tm_kv,
                     const __grid_constant__ CUtensorMap tm_q) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sQ = smem;                      // 9 k-blocks of [64 rows x 64 dims]
  uint8_t *sP = sQ + kQBytes;              // P^T [128 keys x 64 rows]
  uint8_t *sRing = sP + kPBytes;           // kNS slots of 32 KB
  DenseCtrl &c = *reinterpret_cast<DenseCtrl *>(sRing + kNS * kSlotBytes);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // reversed item order: the last shard rows of a request (longest causal
  // ranges) start first, the shortest finish the grid
  const int item = gridDim.x - 1 - blockIdx.x;
  const int row_group = item / a.n_hgroups;
  const int hg = item - row_group * a.n_hgroups;
  const int row0 = row_group * a.g;
  const int h0 = hg * a.hc;
  const int r_valid = a.g * a.hc;

  // ------------------------------------------------------------ setup
  if (tid == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&c.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&c.s_full[s], 1);
      mbar_init(&c.s_free[s], 2 * 128);
    }
    for (int s = 0; s < kFullBars; ++s) mbar_init(&c.full[s], 1);
    mbar_init(&c.p_full, 2 * 128);
    mbar_init(&c.p_free, 1);
    mbar_init(&c.o_full, 1);
    mbar_init(&c.drain[0], 1);
    mbar_init(&c.drain[1], 1);
    mbar_init(&c.q_full, 1);
    c.abort = 0;
    c.need_rescale[0] = c.need_rescale[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&c.tmem_base, kTmemCols);
  if (warp >= 2 && warp < 2 + kProducers && lane == 0) tma_prefetch_desc(&tm_kv);
  if (warp == 1 && lane == 0) tma_prefetch_desc(&tm_q);
  if (tid < kR) {
    c.m_ref[tid] = -INFINITY;
    c.alpha[tid] = 1.f;
  }
  // Per token l of the item (one thread each, in parallel): its global token,
  // valid key range and, merged, whether its shard row owns the token.  The
  // loads form short dependent chains, so they run side by side, not in one
  // thread's loop.
  if (tid < a.g) {
    const int i = row0 + tid;
    int64_t lo = 1, hi = 0;  // empty
    int tok = -1, own = -1;
    if (i < a.n_rows) {
      row_range(a, i, lo, hi);
      if (a.pos[i] + a.kv_start[a.req[i]] > a.s_kv - 1) record_status(a.status, CPMLA_ERR_INDEX);
      tok = a.rows[i];
      if (MERGED) {
        if (tok < 0 || tok >= a.T)
          record_status(a.status, CPMLA_ERR_INDEX);
        else if (a.owner_row[tok] == i)
          own = tok;
        // a row that does not own its token (a replicated decode row outside
        // its owner shard) computes nothing
        if (own < 0) {
          lo = 1;
          hi = 0;
          tok = -1;
        }
      }
    }
    c.tlo[tid] = lo;
    c.thi[tid] = hi;
    c.ttok[tid] = tok;
    c.town[tid] = own;
  }
  __syncthreads();
  // Q rows -> K-major, 128-byte-swizzled k-blocks (zero rows for padding).
  // When an item's tokens start on whole 1 KB swizzle atoms (hc a multiple of
  // 8), each token's hc heads come by TMA, nine boxes of 64 dims landing on
  // q_full, issued once the prologue is done by the first lanes of the eight
  // softmax warps (idle until the first scores; one thread's TMA issues take a
  // few hundred cycles each), while the producers already request the first
  // K tiles; the rows of absent tokens and the padding rows are zeroed by
  // their own thread below.  Otherwise every thread issues all its loads
  // before its first store.
  const bool q_tma = (a.hc & 7) == 0;
  if (q_tma) {
    if (tid == 0) {
      uint32_t bytes = 0;
      for (int l = 0; l < a.g && l * a.hc < r_valid; ++l)
        if (c.ttok[l] >= 0) bytes += (uint32_t)(kKb * a.hc * 128);
      mbar_arrive_expect_tx(&c.q_full, bytes);
    }
  } else {
    constexpr int kPer = kR * (CPMLA_DQK / 8) / kThreads;  // 12 16-byte chunks per thread
    static_assert(kPer * kThreads == kR * (CPMLA_DQK / 8), "Q chunks per thread");
    uint4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int idx = tid + k * kThreads;
      const int r = idx / (CPMLA_DQK / 8);
      const int ch = idx - r * (CPMLA_DQK / 8);
      const int l = r / a.hc, hh = r - l * a.hc;
      v[k] = make_uint4(0, 0, 0, 0);
      if (r < r_valid && c.ttok[l] >= 0)
        v[k] = __ldg(reinterpret_cast<const uint4 *>(a.q + (int64_t)c.ttok[l] * a.q_stride +
                                                     (int64_t)(h0 + hh) * CPMLA_DQK) +
                     ch);
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int idx = tid + k * kThreads;
      const int r = idx / (CPMLA_DQK / 8);
      const int ch = idx - r * (CPMLA_DQK / 8);
      const int kb = ch >> 3, cc = ch & 7;
      *reinterpret_cast<uint4 *>(sQ + kb * (kR * 128) + r * 128 + ((cc ^ (r & 7)) << 4)) = v[k];
    }
  }
  // key range of the item and the tiles that need no mask
  if (tid == 0) {
    int64_t lo_min = INT64_MAX, hi_max = INT64_MIN, lo_max = INT64_MIN, hi_min = INT64_MAX;
    for (int l = 0; l < a.g && row0 + l < a.n_rows; ++l) {
      const int64_t lo = c.tlo[l], hi = c.thi[l];
      lo_max = lo > lo_max ? lo : lo_max;
      hi_min = hi < hi_min ? hi : hi_min;
      if (hi >= lo) {
        lo_min = lo < lo_min ? lo : lo_min;
        hi_max = hi > hi_max ? hi : hi_max;
      }
    }
    if (hi_max < lo_min) {
      c.n_tiles = 0;
      c.tile_lo = 0;
      c.open_lo = c.open_hi = 0;
    } else {
      c.n_tiles = (int)((hi_max - lo_min + kTileKeys) / kTileKeys);
      c.tile_lo = lo_min;
      // tile j is open for every row when 128j >= lo_max - tile_lo and
      // 128j + 127 <= hi_min - tile_lo
      const int64_t a_lo = lo_max - lo_min, a_hi = hi_min - lo_min;
      c.open_lo = (int)((a_lo + kTileKeys - 1) / kTileKeys);
      c.open_hi = a_hi < 0 ? 0 : (int)((a_hi + 1) / kTileKeys);
    }
  }
  __syncthreads();
  if (tid < kR) {
    const int l = tid / a.hc;
    int rlo = 1, rhi = 0;  // empty
    int gt = -1;
    if (tid < r_valid && row0 + l < a.n_rows) {
      const int64_t lo = c.tlo[l], hi = c.thi[l];
      if (hi >= lo) {
        rlo = (int)(lo - c.tile_lo);
        rhi = (int)(hi - c.tile_lo);
      }
      gt = c.town[l];  // merged: the global token row tid writes, if owned
    }
    c.rlo[tid] = rlo;
    c.rhi[tid] = rhi;
    c.gtok[tid] = gt;
    // TMA path: a row that no copy fills (padding, absent token) is zero
    if (q_tma && (tid >= r_valid || c.ttok[l] < 0)) {
#pragma unroll 1
      for (int kb = 0; kb < kKb; ++kb)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          *reinterpret_cast<uint4 *>(sQ + kb * (kR * 128) + tid * 128 + ch * 16) =
              make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();  // Q written by threads, read by tcgen05.mma
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  const int n_tiles = c.n_tiles;
  const uint32_t tO = tmem + 2 * kR;  // O^T chunk c at tO + c*64; S^T buffer b at tmem + b*64
  volatile int *abort = &c.abort;

  // Q copies of the TMA path: box (token l, k-block kb) = number b = 9 l + kb,
  // issued by the first lane of softmax warp b % 8
  if (q_tma && warp >= kSoftmaxWarp0 && lane == 0) {
    const int who = warp - kSoftmaxWarp0;
    for (int b = who; b < kKb * a.g; b += 8) {
      const int l = b / kKb, kb = b - l * kKb;
      if (l * a.hc >= r_valid || c.ttok[l] < 0) continue;
      tma_load_3d(sQ + kb * (kR * 128) + l * a.hc * 128, &tm_q, kb * kKbDims, h0, c.ttok[l],
                  &c.q_full);
    }
  }

  if (warp == 0) {
    // ---------------------------------------------------- score-GEMM issuer
    // takes the K items of the ring sequence
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16(128, kR, 0, 0);
      const uint64_t dq0 = smem_desc(smem_u32(sQ), 16, 1024, kSwz128);
      const uint64_t dr0 = smem_desc(smem_u32(sRing), 16, 1024, kSwz128);
      bool ok = !q_tma || n_tiles == 0 || mbar_wait(&c.q_full, 0, abort, a.status);
      for (int i = 0; i < n_tiles && ok; ++i) {
        const int sb = i & 1;
        if (i >= 2 && !mbar_wait(&c.s_free[sb], ((i >> 1) - 1) & 1, abort, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dS = tmem + sb * kR;
        for (int pr = 0; pr < kKPairs; ++pr) {
          const uint32_t n = ring_pos_k(i, pr), slot = n % kNS;
          if (!mbar_wait(&c.full[n % kFullBars], (n / kFullBars) & 1, abort, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // descriptors advance by (byte offset >> 4) in their address field
          const uint64_t da = dr0 + ((slot * kSlotBytes) >> 4);
          const uint64_t db = dq0 + ((2 * pr * (kR * 128)) >> 4);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (pr == 4 && k >= 4) break;  // the rope pair has one k-block
            const uint32_t h = k >> 2, st = k & 3;
            mma_bf16_ss(dS, da + ((h * kKbBytes + st * 32) >> 4),
                        db + ((h * (kR * 128) + st * 32) >> 4), id_qk,
                        (pr | k) != 0 ? 1u : 0u);
          }
          mma_commit(&c.empty[slot]);
        }
        if (!ok) break;
        mma_commit(&c.s_full[sb]);
      }
      if (!ok) {
        mma_commit(&c.drain[0]);
        drain_wait(&c.drain[0], 0);
      }
      // the Q copies have landed before the CTA can exit
      if (q_tma) drain_wait(&c.q_full, 0);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------- PV-GEMM issuer
    // takes the V items of the ring sequence
    if (lane == 0) {
      constexpr uint32_t id_pv = idesc_bf16(128, kR, 1, 1);
      const uint64_t dp0 = smem_desc(smem_u32(sP), 8192, 1024, kSwz128);
      const uint64_t dr0 = smem_desc(smem_u32(sRing), kKbBytes, 1024, kSwz128);
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        if (!mbar_wait(&c.p_full, j & 1, abort, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ch = 0; ch < kVChunks; ++ch) {
          const uint32_t n = ring_pos_v(j, ch, n_tiles), slot = n % kNS;
          if (!mbar_wait(&c.full[n % kFullBars], (n / kFullBars) & 1, abort, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = dr0 + ((slot * kSlotBytes) >> 4);
#pragma unroll
          for (int st = 0; st < kTileKeys / 16; ++st)
            mma_bf16_ss(tO + ch * kR, da + ((st * 2048) >> 4), dp0 + ((st * 2048) >> 4), id_pv,
                        (j > 0 || st > 0) ? 1u : 0u);
          mma_commit(&c.empty[slot]);
        }
        if (!ok) break;
        mma_commit(&c.p_free);
      }
      mma_commit(&c.o_full);
      if (!ok) {
        mma_commit(&c.drain[1]);
        drain_wait(&c.drain[1], 0);
      }
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 2 + kProducers) {
    // ---------------------------------------------------- producers
    // the ring sequence (see ring_block_base); producer w issues items n
    // with n % kProducers == w - 2
    if (lane == 0) {
      const uint32_t me = warp - 2;
      uint32_t n = 0;
      bool ok = true;
      // item n: K pair / V chunk `it` of `tile` (the same [128 keys x 128]
      // boxes; the rope pair has one k-block)
      auto item = [&](bool is_k, int tile, int it) {
        if (!ok) return;
        if (n % kProducers == me) {
          const uint32_t slot = n % kNS;
          if (n >= (uint32_t)kNS &&
              !mbar_wait(&c.empty[slot], ((n / kNS) - 1) & 1, abort, a.status)) {
            ok = false;
            return;
          }
          const int y = (int)(c.tile_lo + (int64_t)tile * kTileKeys);
          uint8_t *dst = sRing + slot * kSlotBytes;
          const int nkb = (is_k && it == kKPairs - 1) ? 1 : 2;
          uint64_t *fb = &c.full[n % kFullBars];
          mbar_arrive_expect_tx(fb, nkb * kKbBytes);
          tma_load_2d(dst, &tm_kv, it * 128, y, fb);
          if (nkb == 2) tma_load_2d(dst + kKbBytes, &tm_kv, it * 128 + 64, y, fb);
        }
        ++n;
      };
      for (int i = 0; i < 2 && i < n_tiles; ++i)
        for (int p = 0; p < kKPairs; ++p) item(true, i, p);
      for (int t = 0; t < n_tiles && ok; ++t) {
        const bool k = t + 2 < n_tiles;
        for (int ch = 0; ch < kVChunks; ++ch) {
          item(false, t, ch);
          if (k) item(true, t + 2, ch);
        }
        if (k) item(true, t + 2, kKPairs - 1);
      }
      if (!ok) {
        // wait for the loads this thread issued that may still be in flight
        for (uint32_t m = n > (uint32_t)kNS ? n - kNS : 0; m < n; ++m)
          if (m % kProducers == me) drain_wait(&c.full[m % kFullBars], (m / kFullBars) & 1);
      }
    }
    __syncwarp();
  } else if (warp >= kSoftmaxWarp0) {
    // ---------------------------------------------------- softmax + epilogue
    const int wg = (warp - kSoftmaxWarp0) >> 2;
    const int t = tid - kSoftmaxWarp0 * 32 - wg * 128;
    const int q4 = (warp - kSoftmaxWarp0) & 3;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int cbase = wg * kRW;
    const int bar_id = 1 + wg;
    const int open_lo = c.open_lo, open_hi = c.open_hi;
    int seq = 0;
    float l_part[kRW];
#pragma unroll
    for (int r = 0; r < kRW; ++r) l_part[r] = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      if (!group_wait(&c.s_full[sb], (j >> 1) & 1, t, bar_id, c.bflag[wg], seq, abort,
                      a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kRW];
      tmem_ld16(tmem + sb * kR + lane_off + cbase, s);
      tmem_ld16(tmem + sb * kR + lane_off + cbase + 16, s + 16);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&c.s_free[sb]);  // the next-but-one score GEMM may overwrite it
      if (j >= open_lo && j < open_hi) {
#pragma unroll
        for (int r = 0; r < kRW; ++r) s[r] *= a.scale_log2;
      } else {
        const int rel = j * kTileKeys + t;
#pragma unroll
        for (int r = 0; r < kRW; ++r) {
          const bool valid = rel >= c.rlo[cbase + r] && rel <= c.rhi[cbase + r];
          s[r] = valid ? s[r] * a.scale_log2 : -INFINITY;
        }
      }
      {
        float v[kRW];
#pragma unroll
        for (int r = 0; r < kRW; ++r) v[r] = s[r];
        warp_transpose_reduce<kRW, true>(v, lane);
        c.red[wg][q4][lane] = v[0];
      }
      named_bar_sync(bar_id, 128);
      if (t < kRW) {
        const int r = cbase + t;
        const float tile_max = fmaxf(fmaxf(c.red[wg][0][t], c.red[wg][1][t]),
                                     fmaxf(c.red[wg][2][t], c.red[wg][3][t]));
        const float m_old = c.m_ref[r];
        float m_new = m_old;
        if (tile_max > m_old + 8.f) m_new = tile_max;  // lazy move of the reference
        c.alpha[r] = (m_old == -INFINITY) ? 0.f : fast_exp2(m_old - m_new);
        c.m_ref[r] = m_new;
        if (j > 0 && m_new != m_old) c.need_rescale[wg] = j + 1;
      }
      named_bar_sync(bar_id, 128);
      const bool rescale = c.need_rescale[wg] == j + 1;
      uint32_t pk[kRW / 2];
#pragma unroll
      for (int r = 0; r < kRW; r += 2) {
        const float m0 = c.m_ref[cbase + r], m1 = c.m_ref[cbase + r + 1];
        const float p0 = fast_exp2(s[r] - (m0 == -INFINITY ? 0.f : m0));
        const float p1 = fast_exp2(s[r + 1] - (m1 == -INFINITY ? 0.f : m1));
        l_part[r] = l_part[r] * c.alpha[cbase + r] + p0;
        l_part[r + 1] = l_part[r + 1] * c.alpha[cbase + r + 1] + p1;
        pk[r / 2] = pack_bf16x2(p0, p1);
      }
      // PV(j-1) must be done before P^T is overwritten or O^T rescaled
      if (j >= 1 && !group_wait(&c.p_free, (j - 1) & 1, t, bar_id, c.bflag[wg], seq, abort,
                                a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (rescale) {
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
#pragma unroll
          for (int cc = 0; cc < kRW / 16; ++cc) {
            float o[16];
            const uint32_t col = tO + lane_off + ch * kR + cbase + cc * 16;
            tmem_ld16(col, o);
            tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 16; ++x) o[x] *= c.alpha[cbase + cc * 16 + x];
            tmem_st16(col, o);
          }
        }
        tmem_st_wait();
      }
      uint8_t *prow = sP + t * 128;
#pragma unroll
      for (int ch = 0; ch < kRW / 8; ++ch) {
        const int phys = (wg * (kRW / 8) + ch) ^ (t & 7);
        *reinterpret_cast<uint4 *>(prow + phys * 16) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&c.p_full);
    }
    // ------------------------------------------------ epilogue
    if (ok) ok = group_wait(&c.o_full, 0, t, bar_id, c.bflag[wg], seq, abort, a.status);
    if (ok) {
      tc_fence_after();
      warp_transpose_reduce<kRW, false>(l_part, lane);
      c.red[wg][q4][lane] = l_part[0];
      named_bar_sync(bar_id, 128);
      if (t < kRW) {
        const int r = cbase + t;
        const float l = c.red[wg][0][t] + c.red[wg][1][t] + c.red[wg][2][t] + c.red[wg][3][t];
        const float m = c.m_ref[r];
        const bool empty = !(l > 0.f) || m == -INFINITY;
        c.lse[r] = empty ? -INFINITY : (m + __log2f(l)) * 0.69314718055994530942f;
        c.inv_l[r] = empty ? 0.f : 1.f / l;
        float sf = 1.f;
        int64_t ob = -1;
        if (r < r_valid) {
          const int lrow = r / a.hc, hh = r - lrow * a.hc;
          const int i = row0 + lrow;
          if (!MERGED) {
            if (i < a.n_rows) {
              a.lse_part[(int64_t)i * a.H + h0 + hh] = c.lse[r];
              ob = ((int64_t)i * a.H + h0 + hh) * CPMLA_DV;
            }
          } else if (c.gtok[r] >= 0) {
            sf = sink_factor(a.sink, h0 + hh, c.lse[r]);
            a.lse_out[(int64_t)c.gtok[r] * a.H + h0 + hh] = c.lse[r];
          }
        }
        c.sfac[r] = sf;
        c.obase[r] = ob;
      }
      named_bar_sync(bar_id, 128);
      // thread t owns dv t of each O^T chunk; a row's 1/l and sink factor are
      // read once per block of 16 rows (four-wide broadcasts)
      const bool odd = (lane & 1) != 0;
      auto out_block = [&](const float *o, int ch, int cc) {
        float inv[16], sfb[16];
#pragma unroll
        for (int x = 0; x < 16; x += 4) {
          const float4 i4 = *reinterpret_cast<const float4 *>(&c.inv_l[cbase + cc * 16 + x]);
          inv[x] = i4.x;
          inv[x + 1] = i4.y;
          inv[x + 2] = i4.z;
          inv[x + 3] = i4.w;
          if (MERGED) {
            const float4 s4 = *reinterpret_cast<const float4 *>(&c.sfac[cbase + cc * 16 + x]);
            sfb[x] = s4.x;
            sfb[x + 1] = s4.y;
            sfb[x + 2] = s4.z;
            sfb[x + 3] = s4.w;
          }
        }
        if (!MERGED) {
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const int64_t ob = c.obase[cbase + cc * 16 + x];
            if (ob >= 0) a.o_part[ob + ch * 128 + t] = o[x] * inv[x];
          }
        } else {
          // merged: bf16 rows [row][dv] staged in the idle ring (every row:
          // the bulk copies below take only the owned tokens' rows); lane
          // pairs trade one value so that the even lane stores row r at dv
          // t, t+1 and the odd lane row r+1 at dv t-1, t
#pragma unroll
          for (int x = 0; x < 16; x += 2) {
            const int r = cbase + cc * 16 + x;
            // (o / l) x sink factor, rounded as the merge kernel rounds it
            const float v0 = (o[x] * inv[x]) * sfb[x];
            const float v1 = (o[x + 1] * inv[x + 1]) * sfb[x + 1];
            const float got = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
            const uint32_t w = odd ? pack_bf16x2(got, v1) : pack_bf16x2(v0, got);
            // (writing these pairs straight to o_out instead measured 1.416
            // ms against 1.393 for the staged rows and bulk copies)
            *reinterpret_cast<uint32_t *>(sRing + ((size_t)(odd ? r + 1 : r) * CPMLA_DV +
                                                   ch * 128 + (t & ~1)) * 2) = w;
          }
        }
      };
      // O^T chunk ch of this group's rows (32 columns)
      auto load_chunk = [&](int ch, float *o) {
        const uint32_t col = tO + lane_off + ch * kR + cbase;
        tmem_ld16(col, o);
        tmem_ld16(col + 16, o + 16);
      };
      // chunk ch + 1's loads in flight while chunk ch is written (one wait
      // per 32 columns, against one per 16: 1.389 ms against 1.397)
      float oa[kRW], ob[kRW];
      if (n_tiles > 0) {
        load_chunk(0, oa);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int x = 0; x < kRW; ++x) oa[x] = ob[x] = 0.f;
      }
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float *cur = (ch & 1) ? ob : oa;
        float *nxt = (ch & 1) ? oa : ob;
        if (ch < 3 && n_tiles > 0) load_chunk(ch + 1, nxt);
        out_block(cur, ch, 0);
        out_block(cur + 16, ch, 1);
        if (ch < 3 && n_tiles > 0) tmem_ld_wait();
      }
    }
    if (MERGED) {
      // each owned token's hc heads are one contiguous span of o_out: one
      // bulk copy per token from the staged rows, once both warpgroups are
      // here (both always arrive, also after an abort, which skips the copy)
      fence_proxy_async_smem();
      named_bar_sync(3, 2 * 128);
      if (wg == 0 && t == 0 && !*abort) {
        for (int lrow = 0; lrow < a.g && lrow * a.hc < r_valid; ++lrow) {
          const int g = c.gtok[lrow * a.hc];
          if (g < 0) continue;
          bulk_store_s2g(a.o_out + ((int64_t)g * a.H + h0) * CPMLA_DV,
                         sRing + (size_t)lrow * a.hc * CPMLA_DV * 2,
                         (uint32_t)a.hc * CPMLA_DV * 2);
        }
        bulk_commit();
        bulk_wait_read();
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int launch_dense(const AttnArgs &args, const CUtensorMap &tm_kv, const CUtensorMap &tm_q,
                 int n_items, cudaStream_t st) {
  auto kern = args.o_out ? mla_dense_kernel<true> : mla_dense_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return cuda_fail(e, "dense attention: set shared memory size");
  kern<<<n_items, kThreads, kSmem, st>>>(args, tm_kv, tm_q);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "dense attention: launch");
  return CPMLA_OK;
}

}  // namespace cpmla
