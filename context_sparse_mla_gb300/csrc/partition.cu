// partition.cu -- DualChunkSwap partition of a global batch into P virtual
// context-parallel shards (host code).
//
// "[Core] Add MRV2 virtual-batch PCP for MLA", sections "PCP algorithm" and
// "DualChunkSwap partitioning": a prefill request is cut into 2P contiguous
// chunks and shard r takes chunks r and 2P-1-r (PCP=4: {C0,C7}, {C1,C6},
// {C2,C5}, {C3,C4}); each prefill is partitioned on its own; decode rows are
// replicated on every shard.  Readings where the page is silent: uneven chunk
// sizes follow the floor-plus-remainder rule; rows inside a shard go request by
// request, the early chunk before the late one; a decode row is owned by shard 0.
#include <climits>

#include "cpmla_internal.cuh"

namespace {

constexpr int kMaxShards = 1024;

int check_batch(int P, int B, const int32_t *cu, const uint8_t *dec, int64_t *n_total) {
  CPMLA_CHECK_ARG(P >= 1 && P <= kMaxShards, "partition: P=%d outside 1..%d", P, kMaxShards);
  CPMLA_CHECK_ARG(B >= 0, "partition: B=%d < 0", B);
  CPMLA_CHECK_ARG(cu != nullptr, "partition: cu_seqlens is NULL");
  CPMLA_CHECK_ARG(B == 0 || dec != nullptr, "partition: is_decode is NULL");
  CPMLA_CHECK_ARG(cu[0] == 0, "partition: cu_seqlens[0]=%d, expected 0", cu[0]);
  int64_t n = 0;
  for (int b = 0; b < B; ++b) {
    int64_t S = (int64_t)cu[b + 1] - cu[b];
    CPMLA_CHECK_ARG(S >= 0, "partition: cu_seqlens decreases at request %d", b);
    n += dec[b] ? S * P : S;
  }
  CPMLA_CHECK_ARG(n <= INT32_MAX, "partition: %lld shard rows exceed int32", (long long)n);
  *n_total = n;
  return CPMLA_OK;
}

}  // namespace

extern "C" int pcp_partition_size(int P, int B, const int32_t *cu_seqlens,
                                  const uint8_t *is_decode, int64_t *n_rows_total) {
  CPMLA_CHECK_ARG(n_rows_total != nullptr, "pcp_partition_size: n_rows_total is NULL");
  return check_batch(P, B, cu_seqlens, is_decode, n_rows_total);
}

extern "C" int pcp_dualchunk_partition(int P, int B, const int32_t *cu_seqlens,
                                       const int32_t *q_start_pos, const uint8_t *is_decode,
                                       int32_t *shard_offsets, int32_t *rows, int32_t *pos,
                                       int32_t *req, int32_t *owner_shard,
                                       int32_t *owner_row) {
  int64_t n_total = 0;
  int rc = check_batch(P, B, cu_seqlens, is_decode, &n_total);
  if (rc != CPMLA_OK) return rc;
  CPMLA_CHECK_ARG(shard_offsets != nullptr, "pcp_dualchunk_partition: shard_offsets is NULL");
  CPMLA_CHECK_ARG(B == 0 || q_start_pos != nullptr, "pcp_dualchunk_partition: q_start_pos is NULL");
  CPMLA_CHECK_ARG(n_total == 0 || (rows && pos && req),
                  "pcp_dualchunk_partition: rows/pos/req is NULL");
  const int T = B > 0 ? cu_seqlens[B] : 0;
  CPMLA_CHECK_ARG(T == 0 || (owner_shard && owner_row),
                  "pcp_dualchunk_partition: owner arrays are NULL");
  for (int b = 0; b < B; ++b) {
    const int64_t S = cu_seqlens[b + 1] - cu_seqlens[b];
    CPMLA_CHECK_ARG(q_start_pos[b] >= 0 && (int64_t)q_start_pos[b] + S - 1 <= INT32_MAX,
                    "pcp_dualchunk_partition: bad start position %d for request %d",
                    q_start_pos[b], b);
  }
  const int n_chunks = 2 * P;
  int32_t out = 0;
  for (int r = 0; r < P; ++r) {
    shard_offsets[r] = out;
    // the two chunks shard r holds, early one first
    const int mine[2] = {r, n_chunks - 1 - r};
    for (int b = 0; b < B; ++b) {
      const int32_t first = cu_seqlens[b];
      const int32_t S = cu_seqlens[b + 1] - first;
      const int32_t p0 = q_start_pos[b];
      if (is_decode[b]) {
        for (int32_t i = 0; i < S; ++i, ++out) {
          rows[out] = first + i;
          pos[out] = p0 + i;
          req[out] = b;
          if (r == 0) {
            owner_shard[first + i] = 0;
            owner_row[first + i] = out;
          }
        }
        continue;
      }
      const int32_t base = S / n_chunks, extra = S % n_chunks;
      for (int c : mine) {
        const int32_t lo = c * base + (c < extra ? c : extra);
        const int32_t hi = lo + base + (c < extra ? 1 : 0);
        for (int32_t i = lo; i < hi; ++i, ++out) {
          rows[out] = first + i;
          pos[out] = p0 + i;
          req[out] = b;
          owner_shard[first + i] = r;
          owner_row[first + i] = out;
        }
      }
    }
  }
  shard_offsets[P] = out;
  return CPMLA_OK;
}
