// The MoE slot table of one layer, computed by one CTA (blockDim >= N * topk):
// slot 0 is the shared expert (if any), then the distinct routed experts of
// all N tokens in ascending id order; cw[slot][tok] is the token's combine
// weight for that expert (0 where the token does not use it, 1 for the shared
// expert). Ids out of [0, n_experts) are skipped and flagged (status bit 4).
// Used by the routing kernel and by the prep kernel's routing CTA.
#pragma once
#include "bws_common.cuh"
#include "bws_internal.h"

namespace bws {

static BWS_DEV void moe_route_body(const MoeRoute& m) {
  __shared__ int ids[kMaxTokens * kMaxTopk];
  __shared__ int first[kMaxTokens * kMaxTopk];
  const int n = m.N * m.topk;
  const int i = threadIdx.x;
  int bad = 0;
  if (i < n) {
    int e = m.ids[i];
    if (e < 0 || e >= m.n_experts) {
      bad = 1;
      e = -1;
    }
    ids[i] = e;
  }
  bad = __syncthreads_or(bad);
  if (i == 0) m.status[0] = bad ? 4u : 0u;
  for (int s = i; s < m.max_slots * m.N; s += blockDim.x) m.cw[s] = 0.0f;
  __syncthreads();
  if (i < n) {
    int is_first = ids[i] >= 0 ? 1 : 0;
    for (int j = 0; j < i; ++j) is_first &= ids[j] != ids[i];
    first[i] = is_first;
  }
  __syncthreads();
  int rank = 0;
  if (i < n && ids[i] >= 0)
    for (int j = 0; j < n; ++j) rank += (first[j] && ids[j] < ids[i]) ? 1 : 0;
  const int slot = m.has_shared + rank;
  if (i < n && first[i]) m.slot_expert[slot] = ids[i];
  if (i == 0) {
    int c = 0;
    for (int j = 0; j < n; ++j) c += first[j];
    if (m.has_shared) m.slot_expert[0] = -1;
    m.n_slots[0] = c + m.has_shared;
  }
  __syncthreads();   // cw zeroing above is complete
  // ids are distinct per token, so each (slot, token) cell gets one weight
  if (i < n && ids[i] >= 0) m.cw[slot * m.N + i / m.topk] = m.route_w[i];
  if (m.tok_slots != nullptr && i < n) {
    // the token's slots in ascending order (slot order is id order); ids out
    // of range after the valid ones, as -1
    const int t0 = (i / m.topk) * m.topk;
    int pos = 0;
    if (ids[i] >= 0) {
      for (int j = t0; j < t0 + m.topk; ++j) pos += (ids[j] >= 0 && ids[j] < ids[i]) ? 1 : 0;
    } else {
      for (int j = t0; j < t0 + m.topk; ++j) pos += ids[j] >= 0 ? 1 : 0;
      for (int j = t0; j < i; ++j) pos += ids[j] < 0 ? 1 : 0;
    }
    m.tok_slots[t0 + pos] = ids[i] >= 0 ? slot : -1;
  }
  if (m.has_shared && i < m.N) m.cw[i] = 1.0f;
  if (m.ready != nullptr) {   // the table is complete: raise the flag (cumulative over the barrier)
    __syncthreads();
    if (i == 0) store_release(m.ready, 1u);
  }
}

}  // namespace bws
