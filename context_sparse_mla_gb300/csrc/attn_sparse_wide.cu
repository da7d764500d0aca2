// attn_sparse_wide.cu -- top-k sparse partial MLA attention (output + LSE, no
// sink) for one token per CTA, on sm_103a: a bf16 latent KV for up to 64
// heads, or the fp8 KV cache (E4M3 latent with one scale per 128 channels,
// bf16 rope) for 16 heads at a time.
//
// "[DeepSeekV4][PCP] Enable context-parallel prefill for hybrid KV and
// MegaMoE", "Implementation summary": each shard computes the partial
// attention of its query rows over their own top-k keys, merged later by LSE
// (or, for a token's single owner row, in this kernel's epilogue);
// "[Feature][PCP] Add DeepSeek-V4.1-Flash support", "Supported Scope": the
// sparse MLA path with an fp8 KV cache.
//
// One CTA = one token x R heads (bf16: R = 16, 32 or 64; fp8: R = 16).  A token's
// keys are its own, so every gathered key row feeds only this token's heads:
// with R = 64 one CTA covers all heads of a 64-head token and each key row is
// gathered once.
//   * Score GEMM key-major: S^T = K . Q^T, M = 128 keys, N = R, K = 576, into
//     one of two TMEM buffers.  PV GEMM: O^T += V^T . P^T, M = 128 dv x 4
//     chunks, N = R, K = 128 keys, V read from the k-blocks the score GEMM
//     used (the latent is the value, so it stays resident).
//   * Shared memory: Q [R x 576], P^T [128 keys x R], a ring of NP 32 KB pair
//     slots (two k-blocks [128 keys x 64 dims]); pair p of tile j at ring
//     position 4j + p.  R = 16, 32 and fp8: a rope slot of its own and five
//     pair slots, so the rope and pair 0 of tile j+1 need no slot that tile j
//     still holds (bf16 requests them before the softmax of tile j).  R = 64
//     (Q alone is 72 KB): four pair slots, and the rope k-block shares the
//     region of P^T -- the rope of tile j+1 is gathered once the PV GEMM of
//     tile j has read P^T (after the gathers of pair 1), and the score GEMM
//     takes it between pairs 1 and 2.
//   * Gathers: TMA four-row gathers (tile::gather4, 512 B each) issued by the
//     16 softmax warps.  The SM accepts one about every 12-14 cycles and a
//     gather lands ~1,700 (unloaded) to ~3,000 (loaded) cycles after its
//     request; a warp's gather instruction stalls it until the SM has
//     accepted it, so 16 issuing warps keep the queue full (measured: 23
//     B/clk with 8 warps, 42 with 16, 49 with 20).  A tile's slots are freed
//     by the PV GEMM that follows its softmax, so the softmax warps are idle
//     exactly when the next tile's gathers are due.  Warp w of the 16 fills
//     keys 16 (w % 8) .. +15 of k-block w / 8 of every pair slot, and keys
//     8 w .. 8 w + 7 of the rope.  Each warp waits for its slots on its own.
//   * Warp 0 issues the score GEMMs, warps 1 and 2 the PV GEMMs (dv chunks 0,
//     2 and 1, 3): one thread issues an MMA only every ~80 cycles, about the
//     tensor core's time for an N = 64 MMA.  Warp 3 resolves each tile's key
//     rows into shared memory a tile ahead.
//   * Softmax: four warpgroups (warps 4-7, 8-11, 12-15, 16-19) take R/4 score
//     columns each; thread i = TMEM lane i = key i of the tile (dv i of an O^T
//     chunk).  Base 2, with a row reference moved only when a score passes it
//     by 2^8.  Per tile the warps run the gathers of tile j (those the
//     previous softmax unblocked), then its softmax.
//   * fp8 (R = 16, five pair slots, a rope slot of its own): gather warp w
//     fetches the raw E4M3 codes of keys 8 w .. 8 w + 7 of a pair (128 bytes a
//     key, unswizzled, into the upper half of the slot) and, once they have
//     landed, converts them in place to the two fp16 k-blocks of those keys --
//     exactly, since every E4M3 value is an fp16 value.  The score GEMM keeps
//     one accumulator per 128-channel scale group and one for the bf16 rope
//     (five per S^T buffer); Q's latent part is fp16 to meet the fp16 codes.
//     The softmax forms s = rope + sum_g scale_g x group_g, and writes one
//     P^T per dv chunk in fp16 with that chunk's scale folded in, so the PV
//     GEMM also runs on the exact codes.  The five accumulators are
//     independent, so a second thread (warp 20) issues the MMAs of pairs 2
//     and 3 beside warp 0, and each dv chunk of the PV GEMM has its own
//     issuer (warps 1, 2, 21, 22), so a tile's slots free together.
//   * Every wait is bounded.  A wait that decides a warpgroup's control flow
//     is taken by one thread and published to the group, so the group's named
//     barriers always match; a gather warp whose own wait gives up stops
//     gathering.  On expiry the CTA records CPMLA_ERR_TIMEOUT, drains its
//     copies and MMAs, frees TMEM and exits.
#include <cmath>

#include "attn_common.cuh"

namespace cpmla {
namespace {

constexpr int kWThreads = 640;       // 20 warps
constexpr int kWMetaWarp = 3;        // key-row resolution
constexpr int kWGroup0 = 4;          // softmax + gather warps 4..19
constexpr int kWGroups = 4;          // softmax warpgroups
constexpr int kWGatherWarps = 16;
constexpr int kWSoftmaxThreads = 128 * kWGroups;
constexpr int kWSlotBytes = 2 * kKbBytes;  // 32 KB pair slot
constexpr int kWPairs = 4;                 // latent k-block pairs per tile
constexpr int kWRec = 6;                   // gathers remembered per warp for the drain

template <bool FP8, int R>
struct WideCfg {
  static_assert(FP8 ? R == 16 : (R == 16 || R == 32 || R == 64),
                "bf16: 16, 32 or 64 heads per CTA; fp8: 16");
  static constexpr int RC = R / kWGroups;            // score columns per softmax warpgroup
  static constexpr int NS = FP8 ? 5 : 1;             // score accumulators per S^T buffer
  static constexpr bool kRopeInP = !FP8 && R == 64;  // rope shares the P^T region
  static constexpr int kPBytes = kTileKeys * R * 2;  // one P^T [128 keys x R]
  // fp8: one P^T per dv chunk
  static constexpr int kPRegion = FP8 ? 4 * kPBytes : (kRopeInP ? kKbBytes : kPBytes);
  static constexpr int kRopeSlot = kRopeInP ? 0 : kKbBytes;
  static constexpr int kQBytes = R * CPMLA_DQK * 2;
  static constexpr int kPvIssuers = FP8 ? 4 : 2;
  // fp8: warp 20 (second score issuer), warps 21-22 (PV issuers 2-3)
  static constexpr int kThreads = FP8 ? kWThreads + 96 : kWThreads;
  static constexpr uint32_t kTmemCols = 2 * NS * R + 4 * R <= 256 ? 256 : 512;
};
static_assert(WideCfg<false, 64>::kPBytes == kKbBytes, "rope k-block and P^T have one size");
constexpr int kWScore2Warp = 20;  // fp8: second score-GEMM issuer (pairs 2 and 3)
constexpr int kWPv2Warp = 21;     // fp8: PV issuers 2 and 3 (warps 21, 22)

template <bool FP8, int R>
struct WideCtrl {
  uint64_t full[8];       // pair slot ready for the tensor core: one arrival per gather warp
  uint64_t empty[8];      // pair slot released by its PV GEMM chunk
  uint64_t raw[FP8 ? kWGatherWarps : 1][8];  // fp8: a gather warp's codes of a pair slot landed
  uint64_t rope_full;     // rope landed: one arrival per gather warp
  uint64_t rope_empty;    // separate rope slot read by the score GEMM
  uint64_t s_full[2];     // one commit per score issuer
  uint64_t s_free[2];     // S^T buffer read: every softmax thread
  uint64_t p_full;        // P^T written: every softmax thread
  uint64_t p_free;        // PV GEMM of a tile done: every PV issuer
  uint64_t o_full;        // all PV GEMMs done: every PV issuer
  uint64_t drain[8];      // per MMA-issuing thread
  uint64_t meta_full[2];  // key rows of a tile written: the meta warp's 32 lanes
  uint64_t meta_empty[2]; // key rows of a tile no longer needed: every softmax thread
  uint64_t q_full;        // bf16: the token's Q rows landed (TMA)
  uint64_t pv_c0;         // PV issuer 0 has issued dv chunk 0 of a tile
  uint32_t tmem_base;
  int abort;
  int last_slot;          // setup: the largest non-empty top-k slot of the row
  int row_ok;             // setup: the row's token may be read
  int gtok;               // merged output: the global token this CTA writes, or -1
  int bflag[kWGroups][2];  // elected wait results per warpgroup, alternating
  int pf_ok[kWGroups];
  int need_rescale[kWGroups];
  int key_row[2][kTileKeys];  // KV row of each key of a tile, -1 = masked
  // fp8: the four channel-group scales of each key of a tile (0 when masked)
  float4 key_scale[FP8 ? 2 : 1][FP8 ? kTileKeys : 1];
  float red[kWGroups][4][32];
  alignas(16) float m_ref[R];
  alignas(16) float alpha[R];
  float lse[R];
  alignas(16) float inv_l[R];
  alignas(16) float sfac[R];  // merged output: sink factor per head
};

template <bool FP8, int R>
__host__ __device__ constexpr int wide_fixed_bytes() {
  return 1024 + WideCfg<FP8, R>::kQBytes + WideCfg<FP8, R>::kPRegion +
         WideCfg<FP8, R>::kRopeSlot + (int)sizeof(WideCtrl<FP8, R>);
}
// as many pair slots as fit (4 to 8)
template <bool FP8, int R>
__host__ __device__ constexpr int wide_slots() {
  return (232448 - wide_fixed_bytes<FP8, R>()) / kWSlotBytes > 8
             ? 8
             : (232448 - wide_fixed_bytes<FP8, R>()) / kWSlotBytes;
}
template <bool FP8, int R>
__host__ __device__ constexpr int wide_smem_bytes() {
  return wide_fixed_bytes<FP8, R>() + wide_slots<FP8, R>() * kWSlotBytes;
}

constexpr unsigned long long kWDrainLimitNs = 20ull * 1000 * 1000;
__device__ __forceinline__ void wide_drain_wait(uint64_t *bar, uint32_t parity,
                                                unsigned long long limit_ns) {
  unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity) && global_timer_ns() - t0 < limit_ns) {
  }
}

// MERGED: the epilogue writes the token's merged result (AttnArgs::o_out)
// instead of the partial (o_part / lse_part).  tm_q (bf16) is Q as
// [tokens, H, 576]; tm_rope (fp8) is the bf16 rope of the fp8 cache.
template <bool FP8, int R, bool MERGED>
__global__ void __launch_bounds__(WideCfg<FP8, R>::kThreads, 1)
    mla_sparse_wide_kernel(const __grid_constant__ AttnArgs a,
                           const __grid_constant__ CUtensorMap tm_kv,
                           const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_rope) {
  using Cfg = WideCfg<FP8, R>;
  constexpr int RC = Cfg::RC;
  constexpr int NS = Cfg::NS;
  constexpr int NP = wide_slots<FP8, R>();
  static_assert(NP >= kWPairs, "a tile needs four pair slots");
  static_assert(!Cfg::kRopeInP || NP == kWPairs, "the rope-in-P^T order assumes four slots");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sQ = smem;                                 // 9 k-blocks of [R x 64] (fp8: latent fp16)
  uint8_t *sP = sQ + Cfg::kQBytes;                    // P^T (R = 64: also the rope)
  uint8_t *sRope = Cfg::kRopeInP ? sP : sP + Cfg::kPRegion;  // [128 keys x 64 dims]
  uint8_t *sRing = sP + Cfg::kPRegion + Cfg::kRopeSlot;      // NP pair slots
  WideCtrl<FP8, R> &c = *reinterpret_cast<WideCtrl<FP8, R> *>(sRing + NP * kWSlotBytes);

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
      mbar_init(&c.full[s], kWGatherWarps);
      mbar_init(&c.empty[s], 1);
      if (FP8)
        for (int w = 0; w < kWGatherWarps; ++w) mbar_init(&c.raw[w][s], 1);
    }
    mbar_init(&c.rope_full, kWGatherWarps);
    mbar_init(&c.q_full, 1);
    mbar_init(&c.pv_c0, 1);
    mbar_init(&c.rope_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&c.s_full[s], FP8 ? 2 : 1);
      mbar_init(&c.s_free[s], kWSoftmaxThreads);
      mbar_init(&c.meta_full[s], 32);
      mbar_init(&c.meta_empty[s], kWSoftmaxThreads);
    }
    mbar_init(&c.p_full, kWSoftmaxThreads);
    mbar_init(&c.p_free, Cfg::kPvIssuers);
    mbar_init(&c.o_full, Cfg::kPvIssuers);
    for (int s = 0; s < 8; ++s) mbar_init(&c.drain[s], 1);
    c.abort = 0;
    c.last_slot = -1;
    for (int g = 0; g < kWGroups; ++g) c.need_rescale[g] = 0;
    fence_mbar_init();
  }
  if (tid == 32) {
    // the row's token; merged: whether the row owns it (a replicated decode
    // row is computed in every shard and owned by one).  A token outside
    // [0, T) is recorded and the row is treated as empty.
    int ok = row < a.n_rows ? 1 : 0;
    int gt = -1;
    if (ok && MERGED) {
      const int g = a.rows[row];
      if (g < 0 || g >= a.T) {
        record_status(a.status, CPMLA_ERR_INDEX);
        ok = 0;
      } else if (a.owner_row[g] == row) {
        gt = g;
      }
    }
    c.row_ok = ok;
    c.gtok = gt;
  }
  if (warp == 0) tmem_alloc(&c.tmem_base, Cfg::kTmemCols);
  if (warp == kWGroup0 && lane == 0) tma_prefetch_desc(&tm_kv);
  if (warp == 1 && lane == 0) tma_prefetch_desc(FP8 ? &tm_rope : &tm_q);
  if (tid < R) {
    c.m_ref[tid] = -INFINITY;
    c.alpha[tid] = 1.f;
  }
  __syncthreads();
  // Merged: a row that does not own its token (a replicated decode row
  // outside its owner shard) computes nothing.
  const bool row_ok = c.row_ok != 0 && (!MERGED || c.gtok >= 0);
  const int64_t gq = row_ok ? (int64_t)a.rows[row] : -1;
  if (!FP8) {
    // Q rows of this item: nine TMA boxes [R heads x 64 dims] straight into
    // the MMA's K-major, 128-byte-swizzled k-blocks (heads past H read as
    // zero), landing on q_full while the first keys are gathered.  Armed
    // here; the two PV-issuing threads issue the copies once the prologue is
    // done (a thread's TMA issues take a few hundred cycles each, which the
    // prologue would otherwise wait for)
    if (tid == 0 && row_ok) mbar_arrive_expect_tx(&c.q_full, (uint32_t)(kKb * R * 128));
  } else {
    // fp8: Q rows by the threads, the latent part converted to fp16 (it
    // meets fp16 codes in the MMA; the rope part stays bf16 against the bf16
    // rope), into the same K-major, 128-byte-swizzled k-blocks
    constexpr int kChunks = R * (CPMLA_DQK / 8);  // 16-byte chunks
    for (int idx = tid; idx < kChunks; idx += Cfg::kThreads) {
      const int r = idx / (CPMLA_DQK / 8);
      const int ch = idx - r * (CPMLA_DQK / 8);
      uint4 w = make_uint4(0, 0, 0, 0);
      if (row_ok && r < r_valid)
        w = __ldg(reinterpret_cast<const uint4 *>(a.q + gq * a.q_stride +
                                                  (int64_t)(h0 + r) * CPMLA_DQK) +
                  ch);
      if (ch < CPMLA_DV / 8)
        w = make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z),
                       bf16x2_to_f16x2(w.w));
      const int kb = ch >> 3, cc = ch & 7;
      *reinterpret_cast<uint4 *>(sQ + kb * (R * 128) + r * 128 + ((cc ^ (r & 7)) << 4)) = w;
    }
    fence_proxy_async_smem();  // Q written by threads, read by tcgen05.mma
  }
  // the key-row warp's row constants and the list entries of tile 0, loaded
  // beside the scan below instead of after the prologue
  int mw_tpos = 0, mw_lo = 0, mw_hi = 0, mw_len = 0;
  int64_t mw_base = 0;
  const int32_t *mw_lst = nullptr;
  int mw_nxt[4] = {-1, -1, -1, -1};
  if (warp == kWMetaWarp && row_ok) {
    mw_tpos = a.pos[row];
    mw_base = a.kv_start[a.req[row]];
    mw_lst = topk_window(a, row, gq, &mw_len);
    mw_lo = a.kv_lo ? a.kv_lo[row] : 0;
    mw_hi = a.kv_hi ? (a.kv_hi[row] < mw_tpos ? a.kv_hi[row] : mw_tpos) : mw_tpos;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = q * 32 + lane;
      mw_nxt[q] = e < mw_len ? __ldg(mw_lst + e) : -1;
    }
  }
  {
    // the last non-empty slot of the row's list: every thread scans its
    // share (the loads are independent), one shared atomic each
    if (row_ok) {
      int len = 0;
      const int32_t *lst = topk_window(a, row, gq, &len);
      int last = -1;
      for (int e = tid; e < len; e += Cfg::kThreads)
        if (__ldg(lst + e) >= 0) last = e;
      if (last >= 0) atomicMax(&c.last_slot, last);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  const int n_tiles = (c.last_slot + kTileKeys) / kTileKeys;
  // S^T buffer b at tmem + b*NS*R (fp8: accumulator g of it at + g*R, the
  // rope at + 4R); O^T chunk ch at tO + ch*R
  const uint32_t tO = tmem + 2 * NS * R;
  volatile int *abort = &c.abort;

  if (warp == 0 || (FP8 && warp == kWScore2Warp)) {
    // ---------------------------------------------------- score-GEMM issuer(s)
    // bf16: warp 0 issues every MMA of a tile into one accumulator.  fp8:
    // warp 0 the rope and pairs 0-1, warp 20 pairs 2-3, each into its own
    // accumulators; s_full completes when both have committed.
    if (lane == 0) {
      const bool second = FP8 && warp == kWScore2Warp;
      constexpr uint32_t id_rope = idesc_bf16(128, R, 0, 0);
      constexpr uint32_t id_lat = FP8 ? idesc_f16(128, R, 0, 0) : id_rope;
      // descriptors advance by (byte offset >> 4) in their address field
      const uint64_t dq0 = smem_desc(smem_u32(sQ), 16, 1024, kSwz128);
      const uint64_t dr0 = smem_desc(smem_u32(sRing), 16, 1024, kSwz128);
      const uint64_t drope = smem_desc(smem_u32(sRope), 16, 1024, kSwz128);
      const uint64_t dq_rope = dq0 + ((kLatKb * (R * 128)) >> 4);
      const int p_lo = second ? 2 : 0;
      const int p_hi = FP8 ? (second ? 4 : 2) : kWPairs;
      bool ok = FP8 || n_tiles == 0 || mbar_wait(&c.q_full, 0, abort, a.status);
      for (int i = 0; i < n_tiles && ok; ++i) {
        const uint32_t dS = tmem + (i & 1) * NS * R;
        if (i >= 2 && !mbar_wait(&c.s_free[i & 1], ((i >> 1) - 1) & 1, abort, a.status)) {
          ok = false;
          break;
        }
        if (!Cfg::kRopeInP && !second) {
          // the rope first (it starts the accumulator), then its slot is free
          if (!mbar_wait(&c.rope_full, i & 1, abort, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int st = 0; st < 4; ++st)
            mma_bf16_ss(dS + (FP8 ? 4 * R : 0), drope + ((st * 32) >> 4),
                        dq_rope + ((st * 32) >> 4), id_rope, st == 0 ? 0u : 1u);
          mma_commit(&c.rope_empty);
        }
        for (int p = p_lo; p < p_hi; ++p) {
          if (Cfg::kRopeInP && p == 2) {
            // the rope (gathered after pair 1, into the P^T region once the
            // PV GEMM of the previous tile has read it) before the last pairs
            if (!mbar_wait(&c.rope_full, i & 1, abort, a.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int st = 0; st < 4; ++st)
              mma_bf16_ss(dS, drope + ((st * 32) >> 4), dq_rope + ((st * 32) >> 4), id_rope, 1u);
          }
          const uint32_t pos = 4u * i + p, slot = pos % NP;
          if (!mbar_wait(&c.full[slot], (pos / NP) & 1, abort, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = dr0 + ((slot * kWSlotBytes) >> 4);
          const uint64_t db = dq0 + ((2 * p * (R * 128)) >> 4);
          const uint32_t d_acc = FP8 ? dS + p * R : dS;  // fp8: scale group p
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t h = k >> 2, st = k & 3;
            const bool acc = FP8 ? k != 0 : (!Cfg::kRopeInP || (p | k) != 0);
            mma_bf16_ss(d_acc, da + ((h * kKbBytes + st * 32) >> 4),
                        db + ((h * (R * 128) + st * 32) >> 4), id_lat, acc ? 1u : 0u);
          }
        }
        if (!ok) break;
        mma_commit(&c.s_full[i & 1]);
      }
      uint64_t *drain = &c.drain[second ? 1 : 0];
      if (!ok) {
        mma_commit(drain);
        wide_drain_wait(drain, 0, kWaitLimitNs);
      }
      // the Q copy this thread issued has landed before the CTA can exit
      if (!FP8 && row_ok) wide_drain_wait(&c.q_full, 0, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2 || (FP8 && (warp == kWPv2Warp || warp == kWPv2Warp + 1))) {
    // ---------------------------------------------------- PV-GEMM issuers
    // O^T chunk ch += V^T . P^T from tile j's resident pair ch, which is then
    // released.  bf16: issuer `me` takes chunks me and me + 2; fp8: four
    // issuers (warps 1, 2, 21, 22), one chunk each, with the P^T of chunk ch
    // that carries that chunk's scales
    if (lane == 0) {
      const int me = warp <= 2 ? warp - 1 : warp - kWPv2Warp + 2;
      constexpr uint32_t id_pv = FP8 ? idesc_f16(128, R, 1, 1) : idesc_bf16(128, R, 1, 1);
      const uint64_t dp0 = smem_desc(smem_u32(sP), 8192, 8 * PLayout<R>::row_bytes,
                                     PLayout<R>::swz);
      const uint64_t dr0 = smem_desc(smem_u32(sRing), kKbBytes, 1024, kSwz128);
      if (!FP8 && row_ok && me < 2) {
        // bf16: Q's nine boxes, k-blocks me, me + 2, ...
#pragma unroll 1
        for (int kb = me; kb < kKb; kb += 2)
          tma_load_3d(sQ + kb * (R * 128), &tm_q, kb * kKbDims, h0, (int)gq, &c.q_full);
      }
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        if (!mbar_wait(&c.p_full, j & 1, abort, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // chunk 0 reaches the tensor core before the other issuer's first
        // chunk, so the first ring slot of the tile is freed soonest
        if (Cfg::kPvIssuers == 2 && me == 1 && !mbar_wait(&c.pv_c0, j & 1, abort, a.status)) {
          ok = false;
          break;
        }
        for (int ch = me; ch < kWPairs; ch += Cfg::kPvIssuers) {
          const uint32_t slot = (4u * j + ch) % NP;
          const uint64_t da = dr0 + ((slot * kWSlotBytes) >> 4);
          const uint32_t pm = FP8 ? ch * Cfg::kPBytes : 0;
#pragma unroll
          for (int st = 0; st < kTileKeys / 16; ++st)
            mma_bf16_ss(tO + ch * R, da + ((st * 2048) >> 4),
                        dp0 + ((pm + st * 16 * PLayout<R>::row_bytes) >> 4), id_pv,
                        (j > 0 || st > 0) ? 1u : 0u);
          mma_commit(&c.empty[slot]);
          if (Cfg::kPvIssuers == 2 && ch == 0) mbar_arrive(&c.pv_c0);
        }
        mma_commit(&c.p_free);
      }
      mma_commit(&c.o_full);
      if (!ok) {
        mma_commit(&c.drain[2 + me]);
        wide_drain_wait(&c.drain[2 + me], 0, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == kWMetaWarp) {
    // ---------------------------------------------------- key rows
    // key t of tile j: its KV row, or -1 when the slot is empty or outside
    // the row's range (fp8: and its four scales); the list entries of tile
    // j+1 load while tile j's are resolved
    if (row_ok && n_tiles > 0) {
      const int tpos = mw_tpos;
      const int64_t base = mw_base;
      const int len = mw_len;
      const int32_t *lst = mw_lst;
      const int lo = mw_lo, hi = mw_hi;
      int nxt[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) nxt[q] = mw_nxt[q];
      for (int j = 0; j < n_tiles; ++j) {
        int cur[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          cur[q] = nxt[q];
          const int e = (j + 1) * kTileKeys + q * 32 + lane;
          nxt[q] = (j + 1 < n_tiles && e < len) ? __ldg(lst + e) : -1;
        }
        int src[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int p = cur[q];
          src[q] = -1;
          if (p >= 0) {
            if (p > tpos || base + p >= a.s_kv)
              record_status(a.status, CPMLA_ERR_INDEX);
            else if (p >= lo && p <= hi)
              src[q] = (int)(base + p);
          }
        }
        float4 sc[4];
        if (FP8) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            sc[q] = src[q] >= 0 ? __ldg(reinterpret_cast<const float4 *>(a.kv_scale) + src[q])
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // the softmax of tile j-2 (and with it every gather of that tile)
        // must be done with this buffer
        if (j >= 2) {
          int okw = 1;
          if (lane == 0)
            okw = mbar_wait(&c.meta_empty[j & 1], ((j >> 1) - 1) & 1, abort, a.status) ? 1 : 0;
          okw = __shfl_sync(0xffffffffu, okw, 0);
          if (!okw) break;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          c.key_row[j & 1][q * 32 + lane] = src[q];
          if (FP8) c.key_scale[FP8 ? (j & 1) : 0][FP8 ? q * 32 + lane : 0] = sc[q];
        }
        mbar_arrive(&c.meta_full[j & 1]);
      }
    }
    __syncwarp();
  } else if (warp >= kWGroup0 && warp < kWGroup0 + kWGatherWarps) {
    // ---------------------------------------------------- softmax + gathers
    const int gw = warp - kWGroup0;  // gather warp 0..15
    const int grp = gw >> 2;         // softmax warpgroup
    const int q4 = warp & 3;         // TMEM lane quarter this warp may access
    const int t = q4 * 32 + lane;    // key of a tile / dv of a chunk
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int cbase = grp * RC;
    const int bar_id = 1 + grp;
    constexpr int kSpread = 32 / RC;  // lanes sharing one column after a reduction
    int seq = 0;
    bool ok = true;   // the warpgroup goes on (decided group-wide)
    bool gok = true;  // this warp's gathers go on (false once one of its waits gave up)
    float l_part[RC];
#pragma unroll
    for (int r = 0; r < RC; ++r) l_part[r] = 0.f;
    // the last gathers this warp issued, drained if the CTA gives up
    uint64_t *rec_bar[kWRec];
    uint32_t rec_par[kWRec];
    int n_rec = 0;

    // Per-warp bounded wait (lane 0 waits, the warp takes its result).
    auto wwait = [&](uint64_t *bar, uint32_t parity) {
      int r = 1;
      if (lane == 0) r = mbar_wait(bar, parity, abort, a.status) ? 1 : 0;
      gok = __shfl_sync(0xffffffffu, r, 0) != 0;
    };
    // My share of one gather unit.  bf16 pair slot: keys 16 (gw % 8) .. +15
    // of k-block gw / 8 (4 four-row gathers); fp8 pair slot: the raw codes of
    // keys 8 gw .. 8 gw + 7 (2; 128 B a key, unswizzled, in the upper half of
    // the slot); rope: keys 8 gw .. 8 gw + 7 (2).  A masked key fetches KV row
    // 0, which the softmax gives weight exactly 0.
    auto gather = [&](bool rope, int tile, int pr, uint8_t *dst, uint64_t *bar, uint32_t par) {
      const int *krow = c.key_row[tile & 1];
      int k0, n4, x;
      uint8_t *d;
      const CUtensorMap *tm = &tm_kv;
      if (FP8) {
        k0 = 8 * gw;
        n4 = 2;
        d = rope ? dst + gw * 1024 : dst + kKbBytes + gw * 1024;
        x = rope ? 0 : pr * 128;
        if (rope) tm = &tm_rope;
      } else {
        k0 = rope ? 8 * gw : 16 * (gw & 7);
        n4 = rope ? 2 : 4;
        d = rope ? dst + gw * 1024 : dst + (gw >> 3) * kKbBytes + (gw & 7) * 2048;
        x = rope ? CPMLA_DV : pr * 128 + (gw >> 3) * kKbDims;
      }
      if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)n4 * 512);
      __syncwarp();
      if (lane < n4) {
        const int *kr = krow + k0 + 4 * lane;
        tma_gather4(d + lane * 512, tm, x, kr[0] >= 0 ? kr[0] : 0, kr[1] >= 0 ? kr[1] : 0,
                    kr[2] >= 0 ? kr[2] : 0, kr[3] >= 0 ? kr[3] : 0, bar);
      }
      __syncwarp();
      rec_bar[n_rec % kWRec] = bar;
      rec_par[n_rec % kWRec] = par;
      ++n_rec;
    };
    // Pair pr of tile j into its ring slot, once the slot's previous use has
    // been released by its PV GEMM (that tile's softmax is always done by
    // the time this is called).  fp8: the codes land on this warp's own
    // barrier and are converted by convert_pair.
    auto gather_pair = [&](int j, int pr) {
      const int p = 4 * j + pr;
      if (gok && p >= NP) wwait(&c.empty[p % NP], ((p - NP) / NP) & 1);
      if (gok)
        gather(false, j, pr, sRing + (p % NP) * kWSlotBytes,
               FP8 ? &c.raw[FP8 ? gw : 0][p % NP] : &c.full[p % NP], (p / NP) & 1);
    };
    // fp8: this warp's keys of pair pr of tile j, once their codes have
    // landed, converted in place from the raw codes (key k at 16 KB + 128 k)
    // to fp16 in the two 128-byte-swizzled k-blocks; the key's k-block-1 row
    // lies over its own codes, so the warp reads all its codes before it
    // writes.  Unit u of the warp = key 8 gw + u / 8, codes 16 (u % 8) ...
    auto convert_pair = [&](int j, int pr) {
      const int p = 4 * j + pr;
      if (gok) wwait(&c.raw[FP8 ? gw : 0][p % NP], (p / NP) & 1);
      if (!gok) return;
      __syncwarp();
      uint8_t *sl = sRing + (p % NP) * kWSlotBytes;
      uint4 w4[2];
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int u = lane + 32 * b;
        w4[b] = *reinterpret_cast<const uint4 *>(sl + kKbBytes + (8 * gw + (u >> 3)) * 128 +
                                                 (u & 7) * 16);
      }
      __syncwarp();
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int u = lane + 32 * b;
        const int key = 8 * gw + (u >> 3), c8 = u & 7;
        const uint32_t w[4] = {w4[b].x, w4[b].y, w4[b].z, w4[b].w};
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
      fence_proxy_async_smem();  // written by threads, read by tcgen05.mma
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.full[p % NP]);
    };
    auto gather_meta = [&](int j) {
      if (gok) wwait(&c.meta_full[j & 1], (j >> 1) & 1);
    };
    // rope of tile j: its own slot (R = 32, fp8; read first by the score GEMM
    // of tile j-1), or the P^T region once PV(j-1) is done (R = 64)
    auto gather_rope = [&](int j) {
      if (j >= 1 && gok) {
        if (Cfg::kRopeInP)
          wwait(&c.p_free, (j - 1) & 1);
        else
          wwait(&c.rope_empty, (j - 1) & 1);
      }
      if (gok) gather(true, j, 0, sRope, &c.rope_full, j & 1);
    };

    // TMEM columns of this warpgroup (RC of them) without the wait
    auto ld_cols_nw = [&](uint32_t col, float *v) {
      if (RC == 16) {
        tmem_ld16(col, v);
      } else if (RC == 8) {
        tmem_ld8(col, v);
      } else {
        tmem_ld4(col, v);
      }
    };
    auto st_cols = [&](uint32_t col, const float *v) {
      if (RC == 16) {
        tmem_st16(col, v);
      } else if (RC == 8) {
        tmem_st8(col, v);
      } else {
        tmem_st4(col, v);
      }
    };
    auto ld_cols = [&](uint32_t col, float *v) {
      ld_cols_nw(col, v);
      tmem_ld_wait();
    };
    // P^T row of key t, this group's RC columns, 16-byte chunks swizzled
    auto store_p = [&](uint8_t *pbase, const uint32_t *pk) {
      uint8_t *prow = pbase + t * PLayout<R>::row_bytes;
      if (RC >= 8) {
#pragma unroll
        for (int ch = 0; ch < RC / 8; ++ch) {
          const int phys = (grp * (RC / 8) + ch) ^ PLayout<R>::chunk_xor(t);
          *reinterpret_cast<uint4 *>(prow + phys * 16) =
              make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        }
      } else {
        // four columns: half of a 16-byte chunk
        const int phys = (grp >> 1) ^ PLayout<R>::chunk_xor(t);
        *reinterpret_cast<uint2 *>(prow + phys * 16 + (grp & 1) * 8) = make_uint2(pk[0], pk[1]);
      }
    };

    // Softmax of tile j for this warpgroup's columns; false when the CTA
    // gave up.
    auto softmax = [&](int j) -> bool {
      const int sb = j & 1;
      if (!group_wait(&c.s_full[sb], (j >> 1) & 1, t, bar_id, c.bflag[grp], seq, abort,
                      a.status))
        return false;
      tc_fence_after();
      const uint32_t tS = tmem + sb * NS * R + lane_off + cbase;
      // x = score * scale * log2(e) - reference (base 2), -inf for a masked
      // key or a padding head; a reference still at -inf gives +inf
      float x[RC];
      float s8[FP8 ? RC : 1];     // fp8: the scores, kept for a move of the reference
      float ksc[4] = {1.f, 1.f, 1.f, 1.f};  // fp8: this key's group scales
      if (!FP8) {
        ld_cols(tS, x);
      } else {
        // s = rope part + sum_g scale_g * (q . E4M3 codes of group g)
        const float4 sc4 = c.key_scale[FP8 ? sb : 0][FP8 ? t : 0];
        ksc[0] = sc4.x;
        ksc[1] = sc4.y;
        ksc[2] = sc4.z;
        ksc[3] = sc4.w;
        float part[4][RC];
        ld_cols_nw(tS + 4 * R, x);
#pragma unroll
        for (int g = 0; g < 4; ++g) ld_cols_nw(tS + g * R, part[g]);
        tmem_ld_wait();
#pragma unroll
        for (int r = 0; r < RC; ++r) {
          x[r] += ksc[0] * part[0][r] + ksc[1] * part[1][r] + ksc[2] * part[2][r] +
                  ksc[3] * part[3][r];
          s8[FP8 ? r : 0] = x[r];
        }
      }
      const bool valid = c.key_row[sb][t] >= 0;
      float m[RC];
#pragma unroll
      for (int r = 0; r < RC; r += 4) {
        const float4 m4 = *reinterpret_cast<const float4 *>(&c.m_ref[cbase + r]);
        m[r] = m4.x;
        m[r + 1] = m4.y;
        m[r + 2] = m4.z;
        m[r + 3] = m4.w;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int r = 0; r < RC; ++r) {
        x[r] = (valid && cbase + r < r_valid) ? fmaf(x[r], a.scale_log2, -m[r]) : -INFINITY;
        mx = fmaxf(mx, x[r]);
      }
      // PV(j-1) must be done before P^T is overwritten or O^T rescaled:
      // thread 0 waits, the barrier below publishes its result
      if (t == 0)
        c.pf_ok[grp] = (j == 0 || mbar_wait(&c.p_free, (j - 1) & 1, abort, a.status)) ? 1 : 0;
      // the reference of a row moves only when a score passes it by more than
      // 2^8 (always on its first finite score); otherwise no row maxima
      const bool move = named_bar_or(bar_id, 128, mx > 8.f);
      if (!*reinterpret_cast<volatile int *>(&c.pf_ok[grp])) return false;
      if (move) {
        // the scores again (bf16: from TMEM), for each column's tile maximum
        float v[RC];
        if (FP8) {
#pragma unroll
          for (int r = 0; r < RC; ++r) v[r] = s8[FP8 ? r : 0];
        } else {
          ld_cols(tS, v);
        }
#pragma unroll
        for (int r = 0; r < RC; ++r) {
          v[r] = (valid && cbase + r < r_valid) ? v[r] * a.scale_log2 : -INFINITY;
          x[r] = v[r];
        }
        warp_transpose_reduce<RC, true>(x, lane);
        if ((lane & (kSpread - 1)) == 0) c.red[grp][q4][lane / kSpread] = x[0];
        named_bar_sync(bar_id, 128);
        if (t < RC) {
          const int r = cbase + t;
          const float tile_max = fmaxf(fmaxf(c.red[grp][0][t], c.red[grp][1][t]),
                                       fmaxf(c.red[grp][2][t], c.red[grp][3][t]));
          const float m_old = c.m_ref[r];
          float m_new = m_old;
          if (tile_max > m_old + 8.f) m_new = tile_max;  // lazy move of the reference
          c.alpha[r] = (m_old == -INFINITY) ? 0.f : fast_exp2(m_old - m_new);
          c.m_ref[r] = m_new;
          if (j > 0 && m_new != m_old) c.need_rescale[grp] = j + 1;
        }
        named_bar_sync(bar_id, 128);
#pragma unroll
        for (int r = 0; r < RC; ++r) {
          const float mn = c.m_ref[cbase + r];
          x[r] = v[r] - (mn == -INFINITY ? 0.f : mn);
          l_part[r] *= c.alpha[cbase + r];
        }
      }
      // S^T is read: the next-but-one score GEMM may overwrite it
      tc_fence_before();
      mbar_arrive(&c.s_free[sb]);
      uint32_t pk[RC / 2];
#pragma unroll
      for (int r = 0; r < RC; r += 2) {
        const float p0 = fast_exp2(x[r]);
        const float p1 = fast_exp2(x[r + 1]);
        if (!FP8) pk[r / 2] = pack_bf16x2(p0, p1);
        l_part[r] += p0;
        l_part[r + 1] += p1;
        x[r] = p0;
        x[r + 1] = p1;
      }
      const bool rescale = move && c.need_rescale[grp] == j + 1;
      tc_fence_after();
      if (rescale) {
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          float o[RC];
          const uint32_t col = tO + lane_off + ch * R + cbase;
          ld_cols(col, o);
#pragma unroll
          for (int y = 0; y < RC; ++y) o[y] *= c.alpha[cbase + y];
          st_cols(col, o);
        }
        tmem_st_wait();
      }
      if (!FP8) {
        store_p(sP, pk);
      } else {
        // P^T of dv chunk ch: p times this key's scale of channel group ch,
        // in fp16 (11 significant bits) against the fp16 codes
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
#pragma unroll
          for (int r = 0; r < RC; r += 2)
            pk[r / 2] = pack_f16x2(x[r] * ksc[ch], x[r + 1] * ksc[ch]);
          store_p(sP + ch * Cfg::kPBytes, pk);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&c.p_full);
      mbar_arrive(&c.meta_empty[sb]);  // done with this tile's key rows
      return true;
    };

    // The sequence: tile j's gathers, then its softmax.  Ring position p
    // reuses the slot of position p - NP, released by the PV GEMM of that
    // tile, which follows that tile's softmax -- done one iteration earlier.
    // bf16 with five slots (R = 16, 32): the rope and pair 0 of tile j+1
    // wait for nothing, so they are requested before the softmax of tile j --
    // the warps would otherwise wait there for the score GEMM's tail, and the
    // requests queue behind tile j's own -- and only pairs 1-3 of a tile wait
    // for the PV GEMM of the one before (32 heads: 14.1 ms instead of 14.4).
    // R = 64: the rope goes after pair 1 (the PV GEMM of tile j-1 is done by
    // then), so the score GEMM's tail only waits for pairs 2 and 3.  fp8
    // (five slots too): the rope, then each pair converted once its codes
    // have landed, one pair behind the gathers; requesting tile j+1's first
    // units before the softmax made it slower (84.6 ms instead of 80.5).
    constexpr bool kAhead = !Cfg::kRopeInP && !FP8;
    if (kAhead && n_tiles > 0) {
      gather_meta(0);
      gather_rope(0);
      gather_pair(0, 0);
    }
    for (int j = 0; j < n_tiles && ok; ++j) {
      if (FP8) {
        gather_meta(j);
        gather_rope(j);
        gather_pair(j, 0);
        gather_pair(j, 1);
        convert_pair(j, 0);
        gather_pair(j, 2);
        convert_pair(j, 1);
        gather_pair(j, 3);
        convert_pair(j, 2);
        convert_pair(j, 3);
      } else if (!kAhead) {
        gather_meta(j);
        for (int pr = 0; pr < kWPairs; ++pr) {
          gather_pair(j, pr);
          if (pr == 1) gather_rope(j);
        }
      } else {
        for (int pr = 1; pr < kWPairs; ++pr) gather_pair(j, pr);
      }
      if (kAhead && j + 1 < n_tiles) {
        gather_meta(j + 1);
        gather_rope(j + 1);
        gather_pair(j + 1, 0);
      }
      ok = softmax(j);
    }
    if ((!ok || !gok) && lane == 0) {
      // gathers of this warp that may still be landing; a phase another warp
      // never completed gives up after the short limit
      for (int m = n_rec > kWRec ? n_rec - kWRec : 0; m < n_rec; ++m)
        wide_drain_wait(rec_bar[m % kWRec], rec_par[m % kWRec], kWDrainLimitNs);
    }
    __syncwarp();

    // ------------------------------------------------ epilogue
    if (ok) ok = group_wait(&c.o_full, 0, t, bar_id, c.bflag[grp], seq, abort, a.status);
    if (ok) {
      tc_fence_after();
      warp_transpose_reduce<RC, false>(l_part, lane);
      if ((lane & (kSpread - 1)) == 0) c.red[grp][q4][lane / kSpread] = l_part[0];
      named_bar_sync(bar_id, 128);
      if (t < RC) {
        const int r = cbase + t;
        const float l = c.red[grp][0][t] + c.red[grp][1][t] + c.red[grp][2][t] + c.red[grp][3][t];
        const float m = c.m_ref[r];
        const bool empty = !(l > 0.f) || m == -INFINITY;
        c.lse[r] = empty ? -INFINITY : (m + __log2f(l)) * 0.69314718055994530942f;
        c.inv_l[r] = empty ? 0.f : 1.f / l;
        if (r < r_valid && row_ok) {
          if (!MERGED) {
            a.lse_part[(int64_t)row * a.H + h0 + r] = c.lse[r];
          } else if (c.gtok >= 0) {
            c.sfac[r] = sink_factor(a.sink, h0 + r, c.lse[r]);
            a.lse_out[(int64_t)c.gtok * a.H + h0 + r] = c.lse[r];
          }
        }
      }
      named_bar_sync(bar_id, 128);
      // this group's 1/l and sink factors, read once (four-wide broadcasts)
      float inv[RC], sf[RC];
#pragma unroll
      for (int y = 0; y < RC; y += 4) {
        const float4 i4 = *reinterpret_cast<const float4 *>(&c.inv_l[cbase + y]);
        inv[y] = i4.x;
        inv[y + 1] = i4.y;
        inv[y + 2] = i4.z;
        inv[y + 3] = i4.w;
        const float4 s4 = *reinterpret_cast<const float4 *>(&c.sfac[cbase + y]);
        sf[y] = s4.x;
        sf[y + 1] = s4.y;
        sf[y + 2] = s4.z;
        sf[y + 3] = s4.w;
      }
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        float o[RC];
        if (n_tiles > 0) {
          ld_cols(tO + lane_off + ch * R + cbase, o);
        } else {
#pragma unroll
          for (int y = 0; y < RC; ++y) o[y] = 0.f;
        }
        if (!MERGED) {
#pragma unroll
          for (int y = 0; y < RC; ++y) {
            const int r = cbase + y;
            if (r >= r_valid || !row_ok) continue;
            a.o_part[((int64_t)row * a.H + h0 + r) * CPMLA_DV + ch * 128 + t] = o[y] * inv[y];
          }
        } else {
          // merged: bf16 pairs of neighbouring dv -- lane pairs trade one
          // value so that the even lane stores head r at dv t, t+1 and the
          // odd lane head r+1 at dv t-1, t (4-byte stores; a warp writes two
          // 64-byte spans per instruction)
          const bool odd = (lane & 1) != 0;
          const bool own = row_ok && c.gtok >= 0;
#pragma unroll
          for (int y = 0; y < RC; y += 2) {
            const int r = cbase + y;
            const float v0 = r < r_valid ? (o[y] * inv[y]) * sf[y] : 0.f;
            const float v1 = r + 1 < r_valid ? (o[y + 1] * inv[y + 1]) * sf[y + 1] : 0.f;
            const float got = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
            const int hr = odd ? r + 1 : r;
            if (own && hr < r_valid) {
              const uint32_t w = odd ? pack_bf16x2(got, v1) : pack_bf16x2(v0, got);
              *reinterpret_cast<uint32_t *>(a.o_out + ((int64_t)c.gtok * a.H + h0 + hr) * CPMLA_DV +
                                            ch * 128 + (t & ~1)) = w;
            }
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

template <bool FP8, int R, bool MERGED>
int launch_wide_t(const AttnArgs &args, const CUtensorMap &tm_kv, const CUtensorMap &tm_q,
                  const CUtensorMap &tm_rope, int n_items, cudaStream_t stream) {
  constexpr int smem = wide_smem_bytes<FP8, R>();
  static_assert(smem <= 232448, "shared memory budget");
  auto kern = mla_sparse_wide_kernel<FP8, R, MERGED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention: set shared memory size");
  kern<<<n_items, WideCfg<FP8, R>::kThreads, smem, stream>>>(args, tm_kv, tm_q, tm_rope);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention: launch");
  return CPMLA_OK;
}

}  // namespace

int launch_sparse_wide(bool fp8, int R, const AttnArgs &args, const CUtensorMap &tm_kv,
                       const CUtensorMap &tm_q, const CUtensorMap &tm_rope, int n_items,
                       cudaStream_t st) {
  if (fp8) {
    if (R != 16) return fail(CPMLA_ERR_UNSUPPORTED, "sparse attention: fp8 takes 16 heads a CTA");
    return args.o_out ? launch_wide_t<true, 16, true>(args, tm_kv, tm_q, tm_rope, n_items, st)
                      : launch_wide_t<true, 16, false>(args, tm_kv, tm_q, tm_rope, n_items, st);
  }
  if (args.o_out)
    return R == 64   ? launch_wide_t<false, 64, true>(args, tm_kv, tm_q, tm_rope, n_items, st)
           : R == 32 ? launch_wide_t<false, 32, true>(args, tm_kv, tm_q, tm_rope, n_items, st)
                     : launch_wide_t<false, 16, true>(args, tm_kv, tm_q, tm_rope, n_items, st);
  return R == 64   ? launch_wide_t<false, 64, false>(args, tm_kv, tm_q, tm_rope, n_items, st)
         : R == 32 ? launch_wide_t<false, 32, false>(args, tm_kv, tm_q, tm_rope, n_items, st)
                   : launch_wide_t<false, 16, false>(args, tm_kv, tm_q, tm_rope, n_items, st);
}

}  // namespace cpmla
