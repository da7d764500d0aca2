// attn_sparse.cu -- top-k sparse partial MLA attention (output + LSE, no sink)
// for context-parallel prefill, bf16 or fp8 latent KV, on sm_103a.
//
// "[DeepSeekV4][PCP] Enable context-parallel prefill for hybrid KV and
// MegaMoE", "Implementation summary": per-shard partial attention over each
// query's own top-k keys; "[Feature][PCP] Add DeepSeek-V4.1-Flash support",
// "Supported Scope": the sparse MLA path with an fp8 KV cache.
//
// One CTA = one token x up to 32 heads (16 for fp8): its keys are its own, so
// a KV tile serves only that token's heads.
//   * Warps 8-11 gather the token's keys, 128 per tile, into nine 16 KB
//     k-blocks [128 keys x 64 dims], 128-byte swizzled: cp.async for bf16;
//     for fp8, load + exact E4M3 -> bf16 conversion + store (the per-128-
//     channel scales are applied later, so the MMA sees exact values).
//   * Warp 0 issues tcgen05.mma from one thread: S^T = K . Q^T (M = 128 keys,
//     N = R rows, K = 576; fp8 keeps one fp32 accumulator per channel group
//     and one for the rope), then O^T += V^T . P^T (M = 128 dv x 4 chunks,
//     N = R, K = 128 keys).  TMEM holds S^T and O^T.
//   * Warps 4-7 (thread i = key i / dv i of TMEM lane i) apply the scales,
//     mask, run the online softmax with a lazily moved base-2 reference, write
//     P^T (fp8: per chunk, with that chunk's scale, split into high and low
//     bf16 parts) and finally normalise and store O and LSE.
//   * Every wait is bounded; on expiry the CTA records CPMLA_ERR_TIMEOUT,
//     drains its copies and MMAs, and exits.
#include <cmath>

#include "attn_common.cuh"

namespace cpmla {
namespace {

constexpr int kGatherWarp0 = 8;

// Shared-memory control block of the sparse kernel (after the operand buffers).
template <int R>
struct Ctrl {
  uint64_t full[kKb];
  uint64_t empty[kKb];
  uint64_t s_full;
  uint64_t p_full;
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int n_tiles;
  int bflag[3][2];       // elected wait results, per role, alternating slots
  int need_rescale[2];   // per softmax warpgroup: tile index + 1 of the last rescale
  int64_t key_row[2][kTileKeys];  // sparse: global KV row per key, -1 = masked
  float red[2][4][32];
  float m_ref[R];
  float alpha[R];
  float lse[R];
  float inv_l[R];
};

// fp8 keeps eight P^T matrices in a region of their own: per 128-dv chunk,
// P with that chunk's per-key scale folded in, split into a high and a low
// bf16 part.
template <int MODE, int R>
__host__ __device__ constexpr int p_region_bytes() {
  return MODE == kSparseFp8 ? 8 * kTileKeys * R * 2 : 0;
}

template <int MODE, int R>
__host__ __device__ constexpr int smem_bytes() {
  return 1024 /*align slack*/ + R * CPMLA_DQK * 2 + kKb * kKbBytes + p_region_bytes<MODE, R>() +
         (int)sizeof(Ctrl<R>);
}

// Score accumulators: one for bf16 KV; for fp8, one per 128-channel scale
// group plus one for the rope, so the MMA only ever sees exact E4M3 values.
template <int MODE>
__host__ __device__ constexpr int score_accumulators() {
  return MODE == kSparseFp8 ? 5 : 1;
}

template <int MODE, int R>
__global__ void __launch_bounds__(kThreads, 1)
    mla_sparse_kernel(const __grid_constant__ AttnArgs a) {
  // rows handled by one softmax warpgroup, and how many such warpgroups
  constexpr int RW = R < 32 ? R : 32;
  constexpr int NSWG = R / RW;
  static_assert(NSWG == 1, "warps 8-11 gather, so one softmax warpgroup");
  constexpr int NS = score_accumulators<MODE>();
  constexpr int kCols = R * (NS + 4);
  constexpr uint32_t kTmemCols = kCols <= 128 ? 128 : (kCols <= 256 ? 256 : 512);
  static_assert(kCols <= 512, "TMEM budget");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sQ = smem;                       // 9 k-blocks of [R x 64] bf16
  uint8_t *sKV = smem + R * CPMLA_DQK * 2;  // 9 slots of [128 x 64] bf16
  uint8_t *sP = MODE == kSparseFp8 ? sKV + kKb * kKbBytes : sKV + kLatKb * kKbBytes;
  Ctrl<R> &c = *reinterpret_cast<Ctrl<R> *>(sKV + kKb * kKbBytes + p_region_bytes<MODE, R>());

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int item = blockIdx.x;
  const int row_group = item / a.n_hgroups;
  const int hg = item - row_group * a.n_hgroups;
  const int row0 = row_group * a.g;  // first shard row of this CTA
  const int h0 = hg * a.hc;
  const int r_valid = a.g * a.hc;

  // ------------------------------------------------------------ setup
  if (tid == 0) {
    for (int b = 0; b < kKb; ++b) {
      mbar_init(&c.full[b], 128);
      mbar_init(&c.empty[b], 1);
    }
    mbar_init(&c.s_full, 1);
    mbar_init(&c.p_full, 128 * NSWG);
    mbar_init(&c.o_full, 1);
    mbar_init(&c.drain, 1);
    c.abort = 0;
    c.need_rescale[0] = c.need_rescale[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&c.tmem_base, kTmemCols);
  if (tid < R) {
    c.m_ref[tid] = -INFINITY;
    c.alpha[tid] = 1.f;
  }

  // Q rows of this item -> K-major, 128-byte-swizzled k-blocks (zero padding rows)
  for (int idx = tid; idx < R * (CPMLA_DQK / 8); idx += kThreads) {
    const int r = idx / (CPMLA_DQK / 8);
    const int ch = idx - r * (CPMLA_DQK / 8);  // 16-byte chunk along the 576 dims
    const int l = r / a.hc, hh = r - l * a.hc;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < r_valid && row0 + l < a.n_rows) {
      const int64_t gtok = a.rows[row0 + l];
      const uint4 *src = reinterpret_cast<const uint4 *>(a.q + gtok * a.q_stride +
                                                         (int64_t)(h0 + hh) * CPMLA_DQK) +
                         ch;
      v = __ldg(src);
    }
    const int kb = ch >> 3, cc = ch & 7;
    *reinterpret_cast<uint4 *>(sQ + kb * (R * 128) + r * 128 + ((cc ^ (r & 7)) << 4)) = v;
  }

  // number of 128-key tiles of the item
  if (tid == 0) {
    // last non-empty slot of the token's top-k list
    int last = -1;
    if (row0 < a.n_rows) {
      const int32_t *lst = a.topk + (int64_t)a.rows[row0] * a.k;
      for (int e = a.k - 1; e >= 0; --e)
        if (lst[e] >= 0) {
          last = e;
          break;
        }
    }
    c.n_tiles = (last + kTileKeys) / kTileKeys;
  }
  fence_proxy_async_smem();  // Q written by threads, read by tcgen05.mma
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  const int n_tiles = c.n_tiles;
  const uint32_t tS = tmem;           // S^T: NS accumulators of R columns
  const uint32_t tO = tmem + NS * R;  // O^T: 4 chunks of R columns
  volatile int *abort = &c.abort;

  if (warp == 0) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16(128, R, 0, 0);
      constexpr uint32_t id_pv = idesc_bf16(128, R, 1, 1);
      const uint32_t q_base = smem_u32(sQ);
      const uint32_t kv_base = smem_u32(sKV);
      const uint32_t p_base = smem_u32(sP);
      constexpr int p_bytes = kTileKeys * PLayout<R>::row_bytes;  // one P^T matrix
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        const uint32_t par = j & 1;
        // S^T = K_j . Q^T over the 9 k-blocks (latent first, rope last)
        for (int b = 0; b < kKb; ++b) {
          if (!mbar_wait(&c.full[b], par, abort, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // fp8: k-blocks 2g, 2g+1 feed accumulator g, the rope feeds 4
          const uint32_t d_acc = NS == 1 ? tS : tS + (b < kLatKb ? (b >> 1) : 4) * R;
          const bool first_kb = NS == 1 ? b == 0 : (b == kLatKb || (b & 1) == 0);
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint64_t da = smem_desc(kv_base + b * kKbBytes + s * 32, 16, 1024, kSwz128);
            const uint64_t db = smem_desc(q_base + b * (R * 128) + s * 32, 16, 1024, kSwz128);
            mma_bf16_ss(d_acc, da, db, id_qk, (first_kb && s == 0) ? 0u : 1u);
          }
        }
        if (!ok) break;
        mma_commit(&c.s_full);
        // O^T += V_j^T . P_j^T, four 128-dv chunks
        if (!mbar_wait(&c.p_full, par, abort, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
#pragma unroll
          for (int s = 0; s < kTileKeys / 16; ++s) {
            const uint64_t da = smem_desc(kv_base + (2 * ch) * kKbBytes + s * 2048,
                                          kKbBytes /*next 64 dv*/, 1024, kSwz128);
#pragma unroll
            for (int part = 0; part < (MODE == kSparseFp8 ? 2 : 1); ++part) {
              const uint32_t pm = p_base + (MODE == kSparseFp8 ? (2 * ch + part) * p_bytes : 0);
              const uint64_t db = smem_desc(pm + s * 16 * PLayout<R>::row_bytes, 8192,
                                            8 * PLayout<R>::row_bytes, PLayout<R>::swz);
              mma_bf16_ss(tO + ch * R, da, db, id_pv, (j > 0 || s > 0 || part > 0) ? 1u : 0u);
            }
          }
          mma_commit(&c.empty[2 * ch]);
          mma_commit(&c.empty[2 * ch + 1]);
        }
        mma_commit(&c.empty[kLatKb]);
      }
      mma_commit(&c.o_full);
      if (!ok) {
        // let this thread's issued MMAs finish before TMEM and SMEM go away
        mma_commit(&c.drain);
        unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(&c.drain, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4 * NSWG) {
    // ---------------------------------------------------- softmax + epilogue
    // warpgroup wg owns S^T / O^T columns [wg*RW, wg*RW + RW); thread t owns
    // TMEM lane t (key t of a tile, dv t of an O^T chunk)
    const int wg = (warp - kSoftmaxWarp0) >> 2;
    const int t = tid - kSoftmaxWarp0 * 32 - wg * 128;
    const int q4 = (warp - kSoftmaxWarp0) & 3;  // TMEM lane quarter
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int cbase = wg * RW;  // first row (column) of this warpgroup
    const int bar_id = 1 + wg;
    int seq = 0;
    float l_part[RW];
#pragma unroll
    for (int r = 0; r < RW; ++r) l_part[r] = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!group_wait(&c.s_full, j & 1, t, bar_id, c.bflag[wg], seq, abort, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[RW];
      float ksc[4] = {1.f, 1.f, 1.f, 1.f};  // fp8: this key's group scales
      if (NS == 1) {
#pragma unroll
        for (int cc = 0; cc < RW / 16; ++cc)
          tmem_ld16(tS + lane_off + cbase + cc * 16, s + cc * 16);
        tmem_ld_wait();
      } else {
        // s = rope part + sum_g scale_g * (q . e4m3 codes of group g)
        const int64_t src = sparse_key_src(a, row0, j * kTileKeys + t);
        if (src >= 0) {
          const float4 sc4 = __ldg(reinterpret_cast<const float4 *>(a.kv_scale) + src);
          ksc[0] = sc4.x;
          ksc[1] = sc4.y;
          ksc[2] = sc4.z;
          ksc[3] = sc4.w;
        }
#pragma unroll
        for (int cc = 0; cc < RW / 16; ++cc) {
          tmem_ld16(tS + lane_off + 4 * R + cbase + cc * 16, s + cc * 16);
          float part[4][16];
#pragma unroll
          for (int g = 0; g < 4; ++g) tmem_ld16(tS + lane_off + g * R + cbase + cc * 16, part[g]);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 16; ++x)
            s[cc * 16 + x] += ksc[0] * part[0][x] + ksc[1] * part[1][x] + ksc[2] * part[2][x] +
                              ksc[3] * part[3][x];
        }
      }
      // mask, scale to log2 units
      {
        const bool valid = sparse_key_src(a, row0, j * kTileKeys + t) >= 0;
#pragma unroll
        for (int r = 0; r < RW; ++r)
          s[r] = (valid && cbase + r < r_valid) ? s[r] * a.scale_log2 : -INFINITY;
      }
      // row maxima over the tile's 128 keys
      {
        float v[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) v[r] = s[r];
        warp_transpose_reduce<RW, true>(v, lane);
        if (RW == 32 || (lane & 1) == 0) c.red[wg][q4][RW == 32 ? lane : (lane >> 1)] = v[0];
      }
      named_bar_sync(bar_id, 128);
      if (t < RW) {
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
      // p = 2^(s - m_ref); per-lane partial row sums
      // (s is overwritten with p)
      uint32_t pk[RW / 2];
#pragma unroll
      for (int r = 0; r < RW; r += 2) {
        const float m0 = c.m_ref[cbase + r], m1 = c.m_ref[cbase + r + 1];
        const float p0 = fast_exp2(s[r] - (m0 == -INFINITY ? 0.f : m0));
        const float p1 = fast_exp2(s[r + 1] - (m1 == -INFINITY ? 0.f : m1));
        if (NS == 1) pk[r / 2] = pack_bf16x2(p0, p1);
        l_part[r] = l_part[r] * c.alpha[cbase + r] + p0;
        l_part[r + 1] = l_part[r + 1] * c.alpha[cbase + r + 1] + p1;
        s[r] = p0;
        s[r + 1] = p1;
      }
      if (rescale) {
        // O^T columns *= alpha; PV(j-1) is complete (QK(j) was issued after it)
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
#pragma unroll
          for (int cc = 0; cc < RW / 16; ++cc) {
            float o[16];
            const uint32_t col = tO + lane_off + ch * R + cbase + cc * 16;
            tmem_ld16(col, o);
            tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 16; ++x) o[x] *= c.alpha[cbase + cc * 16 + x];
            tmem_st16(col, o);
          }
        }
        tmem_st_wait();
      }
      // this warpgroup's part of P^T row t, into the rope slot (the score
      // GEMM of tile j has consumed it)
#pragma unroll
      for (int m = 0; m < (NS == 1 ? 1 : 8); ++m) {
        uint8_t *prow = sP + m * (kTileKeys * PLayout<R>::row_bytes) + t * PLayout<R>::row_bytes;
        if (NS != 1) {
          // P^T of dv chunk m/2: p times this key's scale of channel group m/2,
          // as a high bf16 part (m even) and the bf16 rounding of the rest (m
          // odd); the PV GEMM adds both, so P reaches the tensor core with ~16
          // significant bits
#pragma unroll
          for (int r = 0; r < RW; r += 2) {
            const float x0 = s[r] * ksc[m >> 1], x1 = s[r + 1] * ksc[m >> 1];
            const uint32_t hi = pack_bf16x2(x0, x1);
            pk[r / 2] = (m & 1) ? pack_bf16x2(x0 - __uint_as_float(hi << 16),
                                              x1 - __uint_as_float(hi & 0xFFFF0000u))
                                : hi;
          }
        }
#pragma unroll
        for (int ch = 0; ch < RW / 8; ++ch) {
          const int logical = wg * (RW / 8) + ch;
          const int phys = logical ^ PLayout<R>::chunk_xor(t);
          *reinterpret_cast<uint4 *>(prow + phys * 16) =
              make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&c.p_full);
    }
    // ------------------------------------------------ epilogue
    if (ok) ok = group_wait(&c.o_full, 0, t, bar_id, c.bflag[wg], seq, abort, a.status);
    if (ok) {
      tc_fence_after();
      warp_transpose_reduce<RW, false>(l_part, lane);
      if (RW == 32 || (lane & 1) == 0) c.red[wg][q4][RW == 32 ? lane : (lane >> 1)] = l_part[0];
      named_bar_sync(bar_id, 128);
      if (t < RW) {
        const int r = cbase + t;
        const float l = c.red[wg][0][t] + c.red[wg][1][t] + c.red[wg][2][t] + c.red[wg][3][t];
        const float m = c.m_ref[r];
        const bool empty = !(l > 0.f) || m == -INFINITY;
        c.lse[r] = empty ? -INFINITY : (m + __log2f(l)) * 0.69314718055994530942f;
        c.inv_l[r] = empty ? 0.f : 1.f / l;
        if (r < r_valid) {
          const int lrow = r / a.hc, hh = r - lrow * a.hc;
          const int i = row0 + lrow;
          if (i < a.n_rows) a.lse_part[(int64_t)i * a.H + h0 + hh] = c.lse[r];
        }
      }
      named_bar_sync(bar_id, 128);
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
#pragma unroll
        for (int cc = 0; cc < RW / 16; ++cc) {
          float o[16];
          if (n_tiles > 0) {
            tmem_ld16(tO + lane_off + ch * R + cbase + cc * 16, o);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int x = 0; x < 16; ++x) o[x] = 0.f;
          }
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const int r = cbase + cc * 16 + x;
            if (r < r_valid) {
              const int lrow = r / a.hc, hh = r - lrow * a.hc;
              const int i = row0 + lrow;
              if (i < a.n_rows)
                a.o_part[((int64_t)i * a.H + h0 + hh) * CPMLA_DV + ch * 128 + t] =
                    o[x] * c.inv_l[r];
            }
          }
        }
      }
    }
  } else if (warp >= kGatherWarp0) {
    // ---------------------------------------------------- sparse gather producer
    const int t = tid - kGatherWarp0 * 32;
    const int row = row0;
    const int64_t gtok = a.rows[row];
    const int32_t *lst = a.topk + gtok * a.k;
    const int tpos = a.pos[row];
    const int64_t base = a.kv_start[a.req[row]];
    int seq = 0;
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      // validity and source row of key t of this tile.  Slot j&1 was last read
      // by the softmax of tile j-2, which finished before tile j-1's slots
      // were released, i.e. before this warpgroup got here.
      {
        const int e = j * kTileKeys + t;
        const int p = e < a.k ? lst[e] : -1;
        if (p >= 0 && (p > tpos || base + p >= a.s_kv)) record_status(a.status, CPMLA_ERR_INDEX);
        c.key_row[j & 1][t] = sparse_key_src(a, row, e);
      }
      named_bar_sync(3, 128);
      for (int b = 0; b < kKb; ++b) {
        if (j > 0 &&
            !group_wait(&c.empty[b], (j - 1) & 1, t, 3, c.bflag[2], seq, abort, a.status)) {
          ok = false;
          break;
        }
        uint8_t *slot = sKV + b * kKbBytes;
        // 128 keys x 8 chunks of 16 B; a warp covers 4 keys x 128 B per step
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int key = it * 16 + (t >> 3);
          const int cc = t & 7;
          const int64_t src = c.key_row[j & 1][key];
          uint8_t *dst = slot + key * 128 + ((cc ^ (key & 7)) << 4);
          if (MODE == kSparseBf16 || b == kLatKb) {
            const __nv_bfloat16 *gp;
            if (MODE == kSparseBf16)
              gp = a.kv + (src >= 0 ? src : 0) * CPMLA_DQK + b * kKbDims + cc * 8;
            else
              gp = a.kv_rope + (src >= 0 ? src : 0) * CPMLA_DROPE + cc * 8;
            cp_async_16(dst, gp, src >= 0 ? 16u : 0u);
          } else {
            // fp8 latent: 8 codes -> 8 bf16, exactly (every E4M3 value is a
            // bf16 value); the group scales are applied to the scores and to
            // P^T instead
            uint4 outv = make_uint4(0, 0, 0, 0);
            if (src >= 0) {
              const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(
                  a.kv8 + src * CPMLA_DV + b * kKbDims + cc * 8));
              const float2 f0 = e4m3x2_to_float2((uint16_t)(raw.x & 0xFFFFu));
              const float2 f1 = e4m3x2_to_float2((uint16_t)(raw.x >> 16));
              const float2 f2 = e4m3x2_to_float2((uint16_t)(raw.y & 0xFFFFu));
              const float2 f3 = e4m3x2_to_float2((uint16_t)(raw.y >> 16));
              outv = make_uint4(pack_bf16x2(f0.x, f0.y), pack_bf16x2(f1.x, f1.y),
                                pack_bf16x2(f2.x, f2.y), pack_bf16x2(f3.x, f3.y));
            }
            *reinterpret_cast<uint4 *>(dst) = outv;
          }
        }
        cp_async_commit();
        // k-block b-1 has landed: publish it to the tensor core
        if (b > 0) {
          cp_async_wait<1>();
          fence_proxy_async_smem();
          mbar_arrive(&c.full[b - 1]);
        }
      }
      if (!ok) break;
      cp_async_wait<0>();
      fence_proxy_async_smem();
      mbar_arrive(&c.full[kKb - 1]);
    }
    cp_async_wait<0>();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}


template <int MODE, int R>
int launch_t(const AttnArgs &args, int n_items, cudaStream_t stream) {
  constexpr int smem = smem_bytes<MODE, R>();
  static_assert(smem <= 232448, "shared memory budget");
  auto kern = mla_sparse_kernel<MODE, R>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention: set shared memory size");
  kern<<<n_items, kThreads, smem, stream>>>(args);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention: launch");
  return CPMLA_OK;
}

}  // namespace

int launch_sparse(int mode, int R, const AttnArgs &args, int n_items, cudaStream_t st) {
  if (mode == kSparseFp8) return launch_t<kSparseFp8, 16>(args, n_items, st);
  return R == 16 ? launch_t<kSparseBf16, 16>(args, n_items, st)
                 : launch_t<kSparseBf16, 32>(args, n_items, st);
}

}  // namespace cpmla
