// attn_sparse.cu -- top-k sparse partial MLA attention (output + LSE, no sink)
// for context-parallel prefill, bf16 or fp8 latent KV, on sm_103a.
//
// "[DeepSeekV4][PCP] Enable context-parallel prefill for hybrid KV and
// MegaMoE", "Implementation summary": per-shard partial attention over each
// query's own top-k keys, merged later by LSE; "[Feature][PCP] Add
// DeepSeek-V4.1-Flash support", "Supported Scope": the sparse MLA path with an
// fp8 KV cache.
//
// One CTA = one token x up to 32 heads (16 for fp8): its keys are its own, so
// a KV tile serves only that token's heads.  The gather is the scarce
// resource, so every key row is gathered once: the latent k-blocks stay
// resident from the score GEMM to the PV GEMM.
//   * Score GEMM key-major: S^T = K . Q^T, M = 128 keys, N = R rows, K = 576,
//     into one of two TMEM buffers.  fp8 keeps one fp32 accumulator per
//     128-channel scale group and one for the rope, so the MMA only sees exact
//     E4M3 values.  PV GEMM: O^T += V^T . P^T, M = 128 dv x 4 chunks, N = R,
//     K = 128 keys, reading V from the same k-blocks.
//   * fp8 computes its latent GEMMs in fp16: E4M3 -> fp16 is one exact
//     conversion per two codes (bf16 takes four), and P^T in fp16 keeps 11
//     significant bits in one matrix per dv chunk.  The latent part of q is
//     rounded to fp16 once (exact for 2^-14 <= |q| < 65504); the rope GEMM
//     stays bf16.
//   * Shared memory holds a ring of 32 KB pair slots (two k-blocks
//     [128 keys x 64 dims] each) and one rope slot.  Pair p of tile j sits at
//     ring position 4j + p, so with five or more slots the first pairs of tile
//     j+1 are gathered while tile j still holds its four.
//   * Gather: warps 8-11 resolve each tile's 128 key rows (and fp8 scales)
//     into shared memory; the rope and the pairs then arrive by TMA four-row
//     gathers (tile::gather4), each 128-byte row landing in the MMA's
//     128-byte-swizzled layout.  One warp issues its gathers one lane at a
//     time, so gather throughput grows with the number of issuing warps:
//     bf16 uses six (2-3 and 8-11), fp8 four (8-11).  fp8 codes land raw
//     in the upper half of their pair slot; warps 2, 3 and 12
//     convert them in place, exactly, to fp16 and release the slot to the
//     tensor core.
//   * MMA issue: one thread issues an MMA only every ~80 cycles, while the
//     tensor core finishes an N = 32 MMA in ~40 (its shared-memory operand
//     reads), so the GEMMs have their own issuing threads: warp 0 the score
//     GEMMs, warp 1 the PV GEMMs (fp8: warps 1 and 13, even and odd dv
//     chunks, since its converter warps leave the softmax more issue slots).
//   * Warps 4-7 (thread i = TMEM lane i = key i / dv i) apply the fp8
//     scales, mask, run the online softmax with a lazily moved base-2
//     reference, write P^T (fp8: per dv chunk with that chunk's scale) and
//     finally normalise and store O and LSE.
//   * Every wait is bounded; on expiry the CTA records CPMLA_ERR_TIMEOUT,
//     drains its copies and MMAs, and exits.
#include <cmath>

#include "attn_common.cuh"

namespace cpmla {
namespace {

constexpr int kGatherWarp0 = 8;
constexpr int kPv2Warp = 13;    // fp8: second PV-GEMM issuer
constexpr int kConverters = 3;  // fp8: converter warps 2, 3, 12

// fp8 adds a converter warp and a second PV issuer
template <int MODE>
__host__ __device__ constexpr int sparse_threads() {
  return MODE == kSparseFp8 ? 448 : kThreads;
}
// converter index of a warp, or -1
__device__ __forceinline__ int converter_index(int warp) {
  return warp == 2 ? 0 : warp == 3 ? 1 : warp == 12 ? 2 : -1;
}
constexpr int kSlotBytes = 2 * kKbBytes;  // 32 KB pair slot
constexpr int kPairs = 4;                 // latent k-block pairs per tile

template <int MODE>
__host__ __device__ constexpr int score_accumulators() {
  return MODE == kSparseFp8 ? 5 : 1;
}

// P^T matrices: one, or for fp8 one per dv chunk (that chunk's scale folded in).
template <int MODE, int R>
__host__ __device__ constexpr int p_region_bytes() {
  return (MODE == kSparseFp8 ? 4 : 1) * kTileKeys * R * 2;
}

template <int MODE, int R>
struct SparseCtrl {
  uint64_t full[8];    // pair slot ready for the tensor core
  uint64_t raw[8];     // fp8: pair slot's codes landed, ready for conversion
  // pair slot released by the PV GEMM: use u of slot s on empty[s][u % 2].
  // Different gather warps fill consecutive uses of a slot, so a warp can
  // wait for use u - 1 to be released before use u - 2 has been; with one
  // barrier per slot the parity test would then pass a phase early.  Use
  // u - 3 has always been released by then (its tile's PV GEMM precedes the
  // softmax that frees the metadata the warp waited for).
  uint64_t empty[8][2];
  uint64_t rope_full;
  uint64_t rope_empty;
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t p_free;
  uint64_t o_full;
  uint64_t drain[3];  // per MMA-issuing thread
  uint64_t meta_full[2];   // key metadata of a tile written (gather -> softmax)
  uint64_t meta_empty[2];  // key metadata of a tile read (softmax -> gather)
  uint32_t tmem_base;
  int abort;
  int n_tiles;
  int bflag[3][2];  // elected wait results (softmax, gather, convert), alternating slots
  int need_rescale;
  int pf_ok;  // the softmax's p_free wait succeeded (thread 0 -> its warpgroup)
  int key_row[2][kTileKeys];  // KV row per key of a tile, -1 = masked
  float4 key_scale[MODE == kSparseFp8 ? 2 : 1][MODE == kSparseFp8 ? kTileKeys : 1];
  float red[4][32];
  float m_ref[R];
  float alpha[R];
  float lse[R];
  float inv_l[R];
  float sfac[R];  // merged output: sink factor per head row
  int gtok;       // merged output: the global token this CTA writes, or -1
};

template <int MODE, int R>
__host__ __device__ constexpr int fixed_bytes() {
  return 1024 + R * CPMLA_DQK * 2 + p_region_bytes<MODE, R>() + kKbBytes /*rope slot*/ +
         (int)sizeof(SparseCtrl<MODE, R>);
}
// as many pair slots as fit (4 to 8)
template <int MODE, int R>
__host__ __device__ constexpr int pair_slots() {
  return (232448 - fixed_bytes<MODE, R>()) / kSlotBytes > 8
             ? 8
             : (232448 - fixed_bytes<MODE, R>()) / kSlotBytes;
}
template <int MODE, int R>
__host__ __device__ constexpr int smem_bytes() {
  return fixed_bytes<MODE, R>() + pair_slots<MODE, R>() * kSlotBytes;
}

// Bounded wait that ignores the abort flag (used to drain own copies and MMAs).
constexpr unsigned long long kDrainLimitNs = 20ull * 1000 * 1000;
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity,
                                           unsigned long long limit_ns = kWaitLimitNs) {
  unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity) && global_timer_ns() - t0 < limit_ns) {
  }
}

// One lane of the warp waits (bounded); the warp takes its result.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int lane,
                                          volatile int *abort, int *status) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(bar, parity, abort, status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// In-place E4M3 -> fp16 conversion of one latent item by the converter
// threads (nthr, a multiple of 32): the raw codes of 128 keys x 128 dims sit
// unswizzled in the upper half of the slot (key k at 16 KB + 128 k); the
// result is two 128-byte-swizzled k-blocks.  Unit u = (key u/8, codes 16
// (u%8) ...); the eight units of a key fall in one warp in the same step,
// and each batch of steps reads all its codes before writing, so every code
// of a key is read before its row is written over it.  One conversion
// instruction per two codes, and exact: every E4M3 value is an fp16 value.
__device__ __forceinline__ void convert_fp8_item(uint8_t *sl, int t, int nthr) {
  constexpr int kUnits = kTileKeys * 8;  // 1024 units of 16 codes
  constexpr int kBatch = 4;              // loads in flight per thread
#pragma unroll 1
  for (int u0 = t; u0 < kUnits; u0 += nthr * kBatch) {
    uint4 raw[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int u = u0 + nthr * b;
      if (u < kUnits)
        raw[b] = *reinterpret_cast<const uint4 *>(sl + kKbBytes + (u >> 3) * 128 + (u & 7) * 16);
    }
    __syncwarp();  // the warp's codes of these keys are read before any row is written
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int u = u0 + nthr * b;
      if (u >= kUnits) continue;
      const int key = u >> 3, c8 = u & 7;
      const uint32_t w[4] = {raw[b].x, raw[b].y, raw[b].z, raw[b].w};
      uint32_t o[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        o[2 * q] = e4m3x2_to_f16x2((uint16_t)(w[q] & 0xFFFFu));
        o[2 * q + 1] = e4m3x2_to_f16x2((uint16_t)(w[q] >> 16));
      }
      // dims 16 c8 .. 16 c8 + 15 of the pair: k-block c8 / 4, chunks 2 (c8 % 4), +1
      const int kb = c8 >> 2, cc0 = 2 * (c8 & 3);
      uint8_t *rowp = sl + kb * kKbBytes + key * 128;
      *reinterpret_cast<uint4 *>(rowp + ((cc0 ^ (key & 7)) << 4)) =
          make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4 *>(rowp + (((cc0 + 1) ^ (key & 7)) << 4)) =
          make_uint4(o[4], o[5], o[6], o[7]);
    }
    __syncwarp();
  }
}

// MERGED: the epilogue writes the token's merged result (AttnArgs::o_out)
// instead of the partial (o_part / lse_part).
template <int MODE, int R, bool MERGED>
__global__ void __launch_bounds__(sparse_threads<MODE>(), 1)
    mla_sparse_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap tm_kv,
                      const __grid_constant__ CUtensorMap tm_rope) {
  static_assert(R == 16 || R == 32, "one softmax warpgroup");
  constexpr int NS = score_accumulators<MODE>();
  constexpr int NP = pair_slots<MODE, R>();
  static_assert(NP >= kPairs, "a tile needs four pair slots");
  constexpr int NT = sparse_threads<MODE>();
  constexpr int kPvIssuers = MODE == kSparseFp8 ? 2 : 1;
  constexpr int kCols = 2 * NS * R + 4 * R;
  constexpr uint32_t kTmemCols = kCols <= 128 ? 128 : (kCols <= 256 ? 256 : 512);
  constexpr int kPBytes = kTileKeys * PLayout<R>::row_bytes;  // one P^T matrix

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sQ = smem;                             // 9 k-blocks of [R x 64] bf16
  uint8_t *sP = sQ + R * CPMLA_DQK * 2;           // P^T matrices
  uint8_t *sRope = sP + p_region_bytes<MODE, R>();  // [128 keys x 64 dims]
  uint8_t *sRing = sRope + kKbBytes;              // NP pair slots
  SparseCtrl<MODE, R> &c = *reinterpret_cast<SparseCtrl<MODE, R> *>(sRing + NP * kSlotBytes);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int item = blockIdx.x;
  const int row = item / a.n_hgroups;  // one shard row (token) per CTA
  const int hg = item - row * a.n_hgroups;
  const int h0 = hg * a.hc;
  const int r_valid = a.hc;

  // ------------------------------------------------------------ setup
  if (tid == 0) {
    for (int s = 0; s < NP; ++s) {
      // bf16: the four half-unit gathers of the pair; fp8: the converter's
      // release after the two half-units of raw codes landed
      mbar_init(&c.full[s], MODE == kSparseFp8 ? 1 : 4);
      mbar_init(&c.raw[s], 2);
      mbar_init(&c.empty[s][0], 1);
      mbar_init(&c.empty[s][1], 1);
    }
    mbar_init(&c.rope_full, 2);  // two half-units
    mbar_init(&c.rope_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&c.s_full[s], 1);
      mbar_init(&c.s_free[s], 128);
      mbar_init(&c.meta_full[s], 128);
      mbar_init(&c.meta_empty[s], 128);
    }
    mbar_init(&c.p_full, 128);
    mbar_init(&c.p_free, kPvIssuers);
    mbar_init(&c.o_full, kPvIssuers);
    for (int s = 0; s < 3; ++s) mbar_init(&c.drain[s], 1);
    c.abort = 0;
    c.need_rescale = 0;
    c.n_tiles = -1;  // the last non-empty slot of the row's list, found below
    fence_mbar_init();
  }
  if (tid == 32) {
    // merged: the global token this CTA writes, if its row owns it (a decode
    // row is computed once per shard, owned by one); beside thread 0's loads
    c.gtok = -1;
    if (MERGED && row < a.n_rows) {
      const int g = a.rows[row];
      if (g < 0 || g >= a.T)
        record_status(a.status, CPMLA_ERR_INDEX);
      else if (a.owner_row[g] == row)
        c.gtok = g;
    }
  }
  if (warp == 0) tmem_alloc(&c.tmem_base, kTmemCols);
  if (tid < R) {
    c.m_ref[tid] = -INFINITY;
    c.alpha[tid] = 1.f;
  }
  __syncthreads();
  // The last non-empty slot of the row's list (every thread scans its share;
  // the loads are independent).  Merged: a row that does not own its token
  // (a replicated decode row outside its owner shard) computes nothing.
  if (row < a.n_rows && (!MERGED || c.gtok >= 0)) {
    int len = 0;
    const int32_t *lst = topk_window(a, row, a.rows[row], &len);
    int last = -1;
    for (int e = tid; e < len; e += NT)
      if (__ldg(lst + e) >= 0) last = e;
    if (last >= 0) atomicMax(&c.n_tiles, last);
  }
  // Q rows of this item -> K-major, 128-byte-swizzled k-blocks (zero padding
  // rows): the token once, then every thread's loads before its stores
  {
    const int64_t gq =
        (row < a.n_rows && (!MERGED || c.gtok >= 0)) ? (int64_t)a.rows[row] : -1;
    constexpr int kChunks = R * (CPMLA_DQK / 8);
    constexpr int kPer = (kChunks + NT - 1) / NT;
    uint4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int idx = tid + k * NT;
      const int r = idx / (CPMLA_DQK / 8);
      const int ch = idx - r * (CPMLA_DQK / 8);
      v[k] = make_uint4(0, 0, 0, 0);
      if (idx < kChunks && r < r_valid && gq >= 0)
        v[k] = __ldg(reinterpret_cast<const uint4 *>(a.q + gq * a.q_stride +
                                                     (int64_t)(h0 + r) * CPMLA_DQK) +
                     ch);
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int idx = tid + k * NT;
      if (idx >= kChunks) continue;
      const int r = idx / (CPMLA_DQK / 8);
      const int ch = idx - r * (CPMLA_DQK / 8);
      uint4 w = v[k];
      // fp8: the latent part meets fp16 codes in the MMA, so it is fp16 too
      // (the rope part stays bf16, against the bf16 rope)
      if (MODE == kSparseFp8 && ch < CPMLA_DV / 8)
        w = make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z),
                       bf16x2_to_f16x2(w.w));
      const int kb = ch >> 3, cc = ch & 7;
      *reinterpret_cast<uint4 *>(sQ + kb * (R * 128) + r * 128 + ((cc ^ (r & 7)) << 4)) = w;
    }
  }
  fence_proxy_async_smem();  // Q written by threads, read by tcgen05.mma
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  const int n_tiles = (c.n_tiles + kTileKeys) / kTileKeys;
  const uint32_t tO = tmem + 2 * NS * R;  // O^T chunk ch at tO + ch*R; S^T buffer b at tmem + b*NS*R
  volatile int *abort = &c.abort;

  if (warp == 0) {
    // ---------------------------------------------------- score-GEMM issuer
    // per tile: the rope (it starts the bf16 accumulator), then pairs 0-3
    // as their slots fill
    if (lane == 0) {
      constexpr uint32_t id_rope = idesc_bf16(128, R, 0, 0);
      constexpr uint32_t id_qk = MODE == kSparseFp8 ? idesc_f16(128, R, 0, 0) : id_rope;
      // descriptors advance by (byte offset >> 4) in their address field
      const uint64_t dq0 = smem_desc(smem_u32(sQ), 16, 1024, kSwz128);
      const uint64_t dr0 = smem_desc(smem_u32(sRing), 16, 1024, kSwz128);
      const uint64_t drope = smem_desc(smem_u32(sRope), 16, 1024, kSwz128);
      bool ok = true;
      for (int i = 0; i < n_tiles && ok; ++i) {
        const uint32_t dS = tmem + (i & 1) * NS * R;
        if (i >= 2 && !mbar_wait(&c.s_free[i & 1], ((i >> 1) - 1) & 1, abort, a.status)) {
          ok = false;
          break;
        }
        if (!mbar_wait(&c.rope_full, i & 1, abort, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        {
          const uint32_t d_acc = NS == 1 ? dS : dS + 4 * R;
#pragma unroll
          for (int st = 0; st < 4; ++st)
            mma_bf16_ss(d_acc, drope + ((st * 32) >> 4),
                        dq0 + ((kLatKb * (R * 128) + st * 32) >> 4), id_rope, st == 0 ? 0u : 1u);
        }
        mma_commit(&c.rope_empty);
        for (int p = 0; p < kPairs; ++p) {
          const uint32_t pos = 4u * i + p, slot = pos % NP;
          if (!mbar_wait(&c.full[slot], (pos / NP) & 1, abort, a.status)) {
            ok = false;
            break;
          }
          // fp8: written through the generic proxy by the converter
          if (MODE == kSparseFp8) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t d_acc = NS == 1 ? dS : dS + p * R;  // fp8: group p
          const uint64_t da = dr0 + ((slot * kSlotBytes) >> 4);
          const uint64_t db = dq0 + ((2 * p * (R * 128)) >> 4);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t h = k >> 2, st = k & 3;
            mma_bf16_ss(d_acc, da + ((h * kKbBytes + st * 32) >> 4),
                        db + ((h * (R * 128) + st * 32) >> 4), id_qk,
                        (NS != 1 && k == 0) ? 0u : 1u);
          }
        }
        if (!ok) break;
        mma_commit(&c.s_full[i & 1]);
      }
      if (!ok) {
        mma_commit(&c.drain[0]);
        drain_wait(&c.drain[0], 0);
      }
    }
    __syncwarp();
  } else if (warp == 1 || (kPvIssuers == 2 && warp == kPv2Warp)) {
    // ---------------------------------------------------- PV-GEMM issuer(s)
    // O^T chunk ch += V^T . P^T from tile j's resident pair ch, which is
    // then released; with two issuers, chunk ch belongs to issuer ch % 2
    if (lane == 0) {
      const int me = warp == 1 ? 0 : 1;
      constexpr uint32_t id_pv = MODE == kSparseFp8 ? idesc_f16(128, R, 1, 1) : idesc_bf16(128, R, 1, 1);
      const uint64_t dp0 = smem_desc(smem_u32(sP), 8192, 8 * PLayout<R>::row_bytes, PLayout<R>::swz);
      const uint64_t dr0 = smem_desc(smem_u32(sRing), kKbBytes, 1024, kSwz128);
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        if (!mbar_wait(&c.p_full, j & 1, abort, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ch = me; ch < kPairs; ch += kPvIssuers) {
          const uint32_t slot = (4u * j + ch) % NP;
          const uint64_t da = dr0 + ((slot * kSlotBytes) >> 4);
          const uint32_t pm = MODE == kSparseFp8 ? ch * kPBytes : 0;
#pragma unroll
          for (int st = 0; st < kTileKeys / 16; ++st)
            mma_bf16_ss(tO + ch * R, da + ((st * 2048) >> 4),
                        dp0 + ((pm + st * 16 * PLayout<R>::row_bytes) >> 4), id_pv,
                        (j > 0 || st > 0) ? 1u : 0u);
          mma_commit(&c.empty[slot][((4u * j + ch) / NP) & 1]);
        }
        mma_commit(&c.p_free);
      }
      mma_commit(&c.o_full);
      if (!ok) {
        mma_commit(&c.drain[1 + me]);
        drain_wait(&c.drain[1 + me], 0);
      }
    }
    __syncwarp();
  } else if (MODE == kSparseFp8 && converter_index(warp) >= 0) {
    // ---------------------------------------------------- fp8 converter
    // pair positions in order: tile j pair p at position 4j + p
    {
      const int t = converter_index(warp) * 32 + lane;
      int seq = 0;
      const uint32_t total = (uint32_t)n_tiles * kPairs;
      for (uint32_t pos = 0; pos < total; ++pos) {
        const uint32_t slot = pos % NP;
        int *f = c.bflag[2] + (seq & 1);
        ++seq;
        if (t == 0) *f = mbar_wait(&c.raw[slot], (pos / NP) & 1, abort, a.status) ? 1 : 0;
        named_bar_sync(4, 32 * kConverters);
        if (!*reinterpret_cast<volatile int *>(f)) break;
        convert_fp8_item(sRing + slot * kSlotBytes, t, 32 * kConverters);
        fence_proxy_async_smem();
        named_bar_sync(4, 32 * kConverters);
        if (t == 0) mbar_arrive(&c.full[slot]);
      }
    }
  } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4) {
    // ---------------------------------------------------- softmax + epilogue
    const int t = tid - kSoftmaxWarp0 * 32;
    const int q4 = warp - kSoftmaxWarp0;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    int seq = 0;
    float l_part[R];
#pragma unroll
    for (int r = 0; r < R; ++r) l_part[r] = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      if (!group_wait(&c.s_full[sb], (j >> 1) & 1, t, 1, c.bflag[0], seq, abort, a.status) ||
          !group_wait(&c.meta_full[sb], (j >> 1) & 1, t, 1, c.bflag[0], seq, abort, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tmem + sb * NS * R + lane_off;
      const int src = c.key_row[sb][t];
      float s[R];
      float ksc[4] = {1.f, 1.f, 1.f, 1.f};  // fp8: this key's group scales
      if (NS == 1) {
#pragma unroll
        for (int cc = 0; cc < R / 16; ++cc) tmem_ld16(tS + cc * 16, s + cc * 16);
        tmem_ld_wait();
      } else {
        // s = rope part + sum_g scale_g * (q . E4M3 codes of group g)
        {
          const float4 sc4 = c.key_scale[sb][t];
          ksc[0] = sc4.x;
          ksc[1] = sc4.y;
          ksc[2] = sc4.z;
          ksc[3] = sc4.w;
        }
#pragma unroll
        for (int cc = 0; cc < R / 16; ++cc) {
          tmem_ld16(tS + 4 * R + cc * 16, s + cc * 16);
          float part[4][16];
#pragma unroll
          for (int g = 0; g < 4; ++g) tmem_ld16(tS + g * R + cc * 16, part[g]);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 16; ++x)
            s[cc * 16 + x] += ksc[0] * part[0][x] + ksc[1] * part[1][x] + ksc[2] * part[2][x] +
                              ksc[3] * part[3][x];
        }
      }
      tc_fence_before();
      mbar_arrive(&c.s_free[sb]);  // the next-but-one score GEMM may overwrite it
      {
        const bool valid = src >= 0;
#pragma unroll
        for (int r = 0; r < R; ++r)
          s[r] = (valid && r < r_valid) ? s[r] * a.scale_log2 : -INFINITY;
      }
      // PV(j-1) must be done before P^T is overwritten or O^T rescaled:
      // thread 0 waits, the barrier below publishes its result
      if (t == 0)
        c.pf_ok = (j == 0 || mbar_wait(&c.p_free, (j - 1) & 1, abort, a.status)) ? 1 : 0;
      // The reference of a row moves only when a score passes it by more than
      // 2^8 (always on the first tile, where it is -inf); otherwise the row
      // maxima are not needed at all.
      bool over = false;
#pragma unroll
      for (int r = 0; r < R; ++r) over |= s[r] > c.m_ref[r] + 8.f;
      const bool move = named_bar_or(1, 128, over);
      if (!*reinterpret_cast<volatile int *>(&c.pf_ok)) {
        ok = false;
        break;
      }
      if (move) {
        {
          float v[R];
#pragma unroll
          for (int r = 0; r < R; ++r) v[r] = s[r];
          warp_transpose_reduce<R, true>(v, lane);
          if (R == 32 || (lane & 1) == 0) c.red[q4][R == 32 ? lane : (lane >> 1)] = v[0];
        }
        named_bar_sync(1, 128);
        if (t < R) {
          const float tile_max =
              fmaxf(fmaxf(c.red[0][t], c.red[1][t]), fmaxf(c.red[2][t], c.red[3][t]));
          const float m_old = c.m_ref[t];
          float m_new = m_old;
          if (tile_max > m_old + 8.f) m_new = tile_max;  // lazy move of the reference
          c.alpha[t] = (m_old == -INFINITY) ? 0.f : fast_exp2(m_old - m_new);
          c.m_ref[t] = m_new;
          if (j > 0 && m_new != m_old) c.need_rescale = j + 1;
        }
        named_bar_sync(1, 128);
      }
      const bool rescale = move && c.need_rescale == j + 1;
      // (s is overwritten with p)
      uint32_t pk[R / 2];
#pragma unroll
      for (int r = 0; r < R; r += 2) {
        const float m0 = c.m_ref[r], m1 = c.m_ref[r + 1];
        const float p0 = fast_exp2(s[r] - (m0 == -INFINITY ? 0.f : m0));
        const float p1 = fast_exp2(s[r + 1] - (m1 == -INFINITY ? 0.f : m1));
        if (NS == 1) pk[r / 2] = pack_bf16x2(p0, p1);
        if (move) {
          l_part[r] = l_part[r] * c.alpha[r] + p0;
          l_part[r + 1] = l_part[r + 1] * c.alpha[r + 1] + p1;
        } else {
          l_part[r] += p0;
          l_part[r + 1] += p1;
        }
        s[r] = p0;
        s[r + 1] = p1;
      }
      tc_fence_after();
      if (rescale) {
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
#pragma unroll
          for (int cc = 0; cc < R / 16; ++cc) {
            float o[16];
            const uint32_t col = tO + lane_off + ch * R + cc * 16;
            tmem_ld16(col, o);
            tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 16; ++x) o[x] *= c.alpha[cc * 16 + x];
            tmem_st16(col, o);
          }
        }
        tmem_st_wait();
      }
#pragma unroll
      for (int m = 0; m < (NS == 1 ? 1 : 4); ++m) {
        uint8_t *prow = sP + m * kPBytes + t * PLayout<R>::row_bytes;
        if (NS != 1) {
          // P^T of dv chunk m: p times this key's scale of channel group m,
          // in fp16 (11 significant bits) against the fp16 codes
#pragma unroll
          for (int r = 0; r < R; r += 2)
            pk[r / 2] = pack_f16x2(s[r] * ksc[m], s[r + 1] * ksc[m]);
        }
#pragma unroll
        for (int ch = 0; ch < R / 8; ++ch) {
          const int phys = ch ^ PLayout<R>::chunk_xor(t);
          *reinterpret_cast<uint4 *>(prow + phys * 16) =
              make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&c.p_full);
      mbar_arrive(&c.meta_empty[sb]);  // done with this tile's key metadata
    }
    // ------------------------------------------------ epilogue
    if (ok) ok = group_wait(&c.o_full, 0, t, 1, c.bflag[0], seq, abort, a.status);
    if (ok) {
      tc_fence_after();
      warp_transpose_reduce<R, false>(l_part, lane);
      if (R == 32 || (lane & 1) == 0) c.red[q4][R == 32 ? lane : (lane >> 1)] = l_part[0];
      named_bar_sync(1, 128);
      if (t < R) {
        const float l = c.red[0][t] + c.red[1][t] + c.red[2][t] + c.red[3][t];
        const float m = c.m_ref[t];
        const bool empty = !(l > 0.f) || m == -INFINITY;
        c.lse[t] = empty ? -INFINITY : (m + __log2f(l)) * 0.69314718055994530942f;
        c.inv_l[t] = empty ? 0.f : 1.f / l;
        if (t < r_valid && row < a.n_rows) {
          if (!MERGED) {
            a.lse_part[(int64_t)row * a.H + h0 + t] = c.lse[t];
          } else if (c.gtok >= 0) {
            c.sfac[t] = sink_factor(a.sink, h0 + t, c.lse[t]);
            a.lse_out[(int64_t)c.gtok * a.H + h0 + t] = c.lse[t];
          }
        }
      }
      named_bar_sync(1, 128);
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
#pragma unroll
        for (int cc = 0; cc < R / 16; ++cc) {
          float o[16];
          if (n_tiles > 0) {
            tmem_ld16(tO + lane_off + ch * R + cc * 16, o);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int x = 0; x < 16; ++x) o[x] = 0.f;
          }
          if (!MERGED) {
#pragma unroll
            for (int x = 0; x < 16; ++x) {
              const int r = cc * 16 + x;
              if (r < r_valid && row < a.n_rows)
                a.o_part[((int64_t)row * a.H + h0 + r) * CPMLA_DV + ch * 128 + t] =
                    o[x] * c.inv_l[r];
            }
          } else if (c.gtok >= 0) {
            // merged: stage bf16 rows [head][dv] in the idle ring, stored below
            __nv_bfloat16 *stage = reinterpret_cast<__nv_bfloat16 *>(sRing);
#pragma unroll
            for (int x = 0; x < 16; ++x) {
              const int r = cc * 16 + x;
              stage[r * CPMLA_DV + ch * 128 + t] =
                  __float2bfloat16_rn((o[x] * c.inv_l[r]) * c.sfac[r]);
            }
          }
        }
      }
      if (MERGED && c.gtok >= 0) {
        // the token's heads h0 .. h0 + r_valid - 1 are one contiguous span of
        // o_out: one bulk copy from the staged rows
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (t == 0) {
          bulk_store_s2g(a.o_out + ((int64_t)c.gtok * a.H + h0) * CPMLA_DV, sRing,
                         (uint32_t)r_valid * CPMLA_DV * 2);
          bulk_commit();
          bulk_wait_read();
        }
      }
    }
  } else {
    // ---------------------------------------------------- gather producers
    // Warps 8-11 resolve each tile's key rows (one key per thread); every
    // issuing warp (bf16: 2-3 and 8-11, fp8: 8-11) then gathers its share of
    // the tile's half-units in order.  A half-unit is 64 keys x one k-block
    // (8 KB): sixteen four-row TMA gathers, one per lane.  Unit order in a
    // tile: rope, then the pairs (bf16: k-block 2p, 2p+1 of pair p; fp8: the
    // raw codes of pair p); half-unit g of the launch-wide sequence belongs
    // to issuing warp g mod the number of issuers.
    constexpr int kIssuers = MODE == kSparseFp8 ? 4 : 6;
    constexpr int kHalves = MODE == kSparseFp8 ? 2 * (1 + kPairs) : 2 * (1 + 2 * kPairs);
    const bool meta = warp >= kGatherWarp0;
    const int widx = meta ? (MODE == kSparseFp8 ? 0 : 2) + warp - kGatherWarp0 : warp - 2;
    const int t = tid - kGatherWarp0 * 32;  // key of a tile (meta warps)
    int tpos = 0, lo = 0, hi = 0, p_next = -1, len = 0;
    int64_t base = 0;
    const int32_t *lst = nullptr;
    if (meta) {
      tpos = a.pos[row];
      base = a.kv_start[a.req[row]];
      lst = topk_window(a, row, a.rows[row], &len);
      lo = a.kv_lo ? a.kv_lo[row] : 0;
      hi = a.kv_hi ? (a.kv_hi[row] < tpos ? a.kv_hi[row] : tpos) : tpos;
      p_next = (n_tiles > 0 && t < len) ? lst[t] : -1;
    }
    int seq = 0;
    bool ok = true;
    // the last half-units this warp issued, drained if the CTA gives up
    constexpr int kRec = 8;
    uint64_t *rec_bar[kRec];
    uint32_t rec_par[kRec];
    int n_rec = 0;
    for (int tile = 0; tile < n_tiles && ok; ++tile) {
      if (meta) {
        // the KV row (and fp8 scales) of key t of this tile; the top-k entry
        // of the next tile is loaded now, to be used one iteration later
        const int p = p_next;
        {
          const int e = (tile + 1) * kTileKeys + t;
          p_next = (tile + 1 < n_tiles && e < len) ? lst[e] : -1;
        }
        int src = -1;
        if (p >= 0) {
          if (p > tpos || base + p >= a.s_kv)
            record_status(a.status, CPMLA_ERR_INDEX);
          else if (p >= lo && p <= hi)
            src = (int)(base + p);
        }
        float4 sc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (MODE == kSparseFp8 && src >= 0)
          sc = __ldg(reinterpret_cast<const float4 *>(a.kv_scale) + src);
        // the softmax of tile-2 must be done with this metadata slot
        if (tile >= 2 && !group_wait(&c.meta_empty[tile & 1], ((tile >> 1) - 1) & 1, t, 3,
                                     c.bflag[1], seq, abort, a.status)) {
          ok = false;
          break;
        }
        c.key_row[tile & 1][t] = src;
        if (MODE == kSparseFp8) c.key_scale[tile & 1][t] = sc;
        mbar_arrive(&c.meta_full[tile & 1]);
      }
      if (!warp_wait(&c.meta_full[tile & 1], (tile >> 1) & 1, lane, abort, a.status)) {
        ok = false;
        break;
      }
      const int *krow = c.key_row[tile & 1];
      const int first = ((widx - (tile * kHalves) % kIssuers) % kIssuers + kIssuers) % kIssuers;
      for (int i = first; i < kHalves; i += kIssuers) {
        const int u = i >> 1, half = i & 1;
        uint64_t *bar;
        uint32_t par;
        uint8_t *dst;
        const CUtensorMap *tm;
        int x;
        if (u == 0) {
          if (tile >= 1 && !warp_wait(&c.rope_empty, (tile - 1) & 1, lane, abort, a.status)) {
            ok = false;
            break;
          }
          bar = &c.rope_full;
          par = tile & 1;
          dst = sRope;
          tm = &tm_rope;
          x = MODE == kSparseBf16 ? CPMLA_DV : 0;
        } else {
          const int pr = MODE == kSparseBf16 ? (u - 1) >> 1 : u - 1;
          const int kb = MODE == kSparseBf16 ? (u - 1) & 1 : 0;
          const uint32_t pos = 4u * tile + pr, slot = pos % NP;
          if (pos >= (uint32_t)NP &&
              !warp_wait(&c.empty[slot][((pos / NP) - 1) & 1], (((pos / NP) - 1) >> 1) & 1, lane,
                         abort, a.status)) {
            ok = false;
            break;
          }
          par = (pos / NP) & 1;
          tm = &tm_kv;
          if (MODE == kSparseBf16) {
            // dims [128 pr + 64 kb, +64) as one 128-byte-swizzled k-block
            bar = &c.full[slot];
            dst = sRing + slot * kSlotBytes + kb * kKbBytes;
            x = pr * 128 + kb * kKbDims;
          } else {
            // raw E4M3 codes of dims [128 pr, 128 pr + 128): 128 B per key,
            // unswizzled, in the upper half of the slot
            bar = &c.raw[slot];
            dst = sRing + slot * kSlotBytes + kKbBytes;
            x = pr * 128;
          }
        }
        if (lane == 0) mbar_arrive_expect_tx(bar, kKbBytes / 2);
        __syncwarp();
        if (lane < 16) {
          // keys 64 half + 4 lane .. +3; a masked key fetches row 0, which
          // the softmax gives weight exactly 0
          const int *kr = krow + half * 64 + 4 * lane;
          tma_gather4(dst + half * (kKbBytes / 2) + lane * 512, tm, x, kr[0] >= 0 ? kr[0] : 0,
                      kr[1] >= 0 ? kr[1] : 0, kr[2] >= 0 ? kr[2] : 0, kr[3] >= 0 ? kr[3] : 0,
                      bar);
        }
        rec_bar[n_rec % kRec] = bar;
        rec_par[n_rec % kRec] = par;
        ++n_rec;
      }
    }
    if (!ok && lane == 0) {
      // gathers of this warp that may still be landing; a phase that another
      // warp never completed gives up after the short limit
      for (int m = n_rec > kRec ? n_rec - kRec : 0; m < n_rec; ++m)
        drain_wait(rec_bar[m % kRec], rec_par[m % kRec], kDrainLimitNs);
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int MODE, int R, bool MERGED>
int launch_t(const AttnArgs &args, const CUtensorMap &tm_kv, const CUtensorMap &tm_rope,
             int n_items, cudaStream_t stream) {
  constexpr int smem = smem_bytes<MODE, R>();
  static_assert(pair_slots<MODE, R>() >= kPairs, "shared memory budget");
  static_assert(smem <= 232448, "shared memory budget");
  auto kern = mla_sparse_kernel<MODE, R, MERGED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention: set shared memory size");
  kern<<<n_items, sparse_threads<MODE>(), smem, stream>>>(args, tm_kv, tm_rope);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention: launch");
  return CPMLA_OK;
}

}  // namespace

int launch_sparse(int mode, int R, const AttnArgs &args, const CUtensorMap &tm_kv,
                  const CUtensorMap &tm_rope, int n_items, cudaStream_t st) {
  if (args.o_out) {
    if (mode == kSparseFp8)
      return launch_t<kSparseFp8, 16, true>(args, tm_kv, tm_rope, n_items, st);
    return R == 16 ? launch_t<kSparseBf16, 16, true>(args, tm_kv, tm_rope, n_items, st)
                   : launch_t<kSparseBf16, 32, true>(args, tm_kv, tm_rope, n_items, st);
  }
  if (mode == kSparseFp8) return launch_t<kSparseFp8, 16, false>(args, tm_kv, tm_rope, n_items, st);
  return R == 16 ? launch_t<kSparseBf16, 16, false>(args, tm_kv, tm_rope, n_items, st)
                 : launch_t<kSparseBf16, 32, false>(args, tm_kv, tm_rope, n_items, st);
}

}  // namespace cpmla
