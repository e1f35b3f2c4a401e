// C ABI of the MXFP4 mixture-of-experts layer.
//
// One layer runs as six kernels on the caller's stream, chained with
// programmatic dependent launch:
//   route   -> slot table: the shared expert, then the distinct routed experts
//              of all N tokens in ascending id order, and each (slot, token)
//              combine weight (0 where the token does not use the expert)
//   prep x  -> the tokens' activations as f16 bands
//   gate/up -> h[slot] = BF16(SiLU(W_gate x) * W_up x) for every live slot
//   prep h  -> h as f16 bands, per (slot, token)
//   down    -> ys[slot] = W_down h[slot] (FP32)
//   combine -> y = sum over slots, in slot order, of cw * ys
// Every expert that any token uses is read exactly once per call.
// In the decode stream the routing runs as one extra CTA of the RMSNorm prep
// before the experts, and the combine is folded into the next RMSNorm prep,
// so an MoE layer there costs four kernels.
#include <cuda_runtime.h>

#include "../../include/bws.h"
#include "bws_abi_util.h"
#include "bws_internal.h"

namespace bws {

struct MoeLayout {
  int max_slots, tiles_gu, tiles_dn, n_tiles, d_pad_x, d_pad_h;
  // two route buffers (n_slots, slot table, combine weights): the decode
  // stream alternates them by layer, so that a layer's routing never
  // overwrites the weights the previous layer's combine still reads
  size_t off_route, off_slot_expert, off_cw, off_status;
  size_t off_route_b, off_slot_expert_b, off_cw_b;
  GemvWorkspace xw;   // offsets relative to off_x
  size_t off_x;
  size_t off_h;
  GemvWorkspace hw;   // offsets relative to off_hp (prep part only)
  size_t off_hp;
  size_t off_ys, off_counters, off_partials, partials_bytes, total;
};

static MoeLayout moe_layout(const bws_moe_layer* L, int N, int topk) {
  MoeLayout m;
  const int has_shared = L->shared_gate_up_codes != nullptr ? 1 : 0;
  m.max_slots = N * topk + has_shared;
  m.tiles_gu = (L->inter + 15) / 16;
  m.tiles_dn = (L->hidden + 31) / 32;
  m.n_tiles = m.max_slots * (m.tiles_gu > m.tiles_dn ? m.tiles_gu : m.tiles_dn);
  size_t o = 0;
  m.off_route = o; o += 256;
  m.off_status = m.off_route + 16;
  m.off_slot_expert = o; o += align256(sizeof(int) * m.max_slots);
  m.off_cw = o; o += align256(sizeof(float) * (size_t)m.max_slots * N);
  m.off_route_b = o; o += 256;
  m.off_slot_expert_b = o; o += align256(sizeof(int) * m.max_slots);
  m.off_cw_b = o; o += align256(sizeof(float) * (size_t)m.max_slots * N);
  m.off_x = o;
  m.xw = gemv_workspace_layout(N, L->hidden, 0, 0, 1);
  o += m.xw.off_counters;   // header, exps, flags, hi, lo
  m.off_h = o; o += align256(2 * (size_t)m.max_slots * N * L->inter);
  m.off_hp = o;
  m.hw = gemv_workspace_layout(N, L->inter, 0, 0, m.max_slots);
  o += m.hw.off_counters;
  m.off_ys = o; o += align256(sizeof(float) * (size_t)m.max_slots * N * L->hidden);
  m.off_counters = o; o += align256(sizeof(uint32_t) * (size_t)m.n_tiles);
  // partial sums of either expert kernel
  m.partials_bytes = sizeof(float) * kSlotFloats * ((size_t)m.n_tiles + gemv_max_warps());
  const size_t pt = moe_tma_partials_bytes(kEpiSwiGLU, L->inter, m.max_slots) >
                            moe_tma_partials_bytes(kEpiStoreF32, L->hidden, m.max_slots)
                        ? moe_tma_partials_bytes(kEpiSwiGLU, L->inter, m.max_slots)
                        : moe_tma_partials_bytes(kEpiStoreF32, L->hidden, m.max_slots);
  if (pt > m.partials_bytes) m.partials_bytes = pt;
  m.off_partials = o; o += align256(m.partials_bytes);
  m.total = o;
  return m;
}

static int check_moe(const bws_moe_layer* L, int N, int topk, const char* name) {
  if (L == nullptr) return fail(BWS_ERR_INVALID_ARG, "%s: null layer descriptor", name);
  if (N < 1 || N > kMaxTokens) return fail(BWS_ERR_INVALID_ARG, "%s: N = %d must be in [1, %d]", name, N, kMaxTokens);
  if (topk < 1 || topk > kMaxTopk) return fail(BWS_ERR_INVALID_ARG, "%s: topk = %d must be in [1, %d]", name, topk, kMaxTopk);
  if (L->n_experts < 1 || L->hidden < 32 || L->hidden % 32 || L->inter < 32 || L->inter % 32)
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: n_experts=%d hidden=%d inter=%d (hidden, inter %% 32 == 0)", name,
                L->n_experts, L->hidden, L->inter);
  if (!L->gate_up_codes || !L->gate_up_scales || !L->down_codes || !L->down_scales)
    return fail(BWS_ERR_INVALID_ARG, "%s: null expert tensor", name);
  const bool sh = L->shared_gate_up_codes != nullptr;
  if (sh && (!L->shared_gate_up_scales || !L->shared_down_codes || !L->shared_down_scales))
    return fail(BWS_ERR_INVALID_ARG, "%s: incomplete shared expert", name);
  if (!aligned(L->gate_up_codes, 16) || !aligned(L->down_codes, 16) || L->gate_up_codes_stride % 16 ||
      L->down_codes_stride % 16 || (sh && (!aligned(L->shared_gate_up_codes, 16) || !aligned(L->shared_down_codes, 16))))
    return fail(BWS_ERR_MISALIGNED, "%s: expert codes and strides must be 16-byte aligned", name);
  const size_t gu_codes = (size_t)2 * L->inter * L->hidden / 2, dn_codes = (size_t)L->hidden * L->inter / 2;
  if (L->gate_up_codes_stride < gu_codes || L->down_codes_stride < dn_codes ||
      L->gate_up_scales_stride < (size_t)2 * L->inter * L->hidden / 32 ||
      L->down_scales_stride < (size_t)L->hidden * L->inter / 32)
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: expert strides smaller than one expert", name);
  return BWS_OK;
}

// gate/up, prep h and down of one MoE layer for the slots of the given slot
// table: ys[slot][tok] = W_down h (FP32) in the workspace.
int enqueue_moe_experts(const bws_moe_layer* L, int N, int topk, const int* n_slots, const int* slot_expert,
                        const XPrep& xp, char* w, cudaStream_t st, const char* name, const uint32_t* ready) {
  const MoeLayout m = moe_layout(L, N, topk);
  uint32_t* counters = reinterpret_cast<uint32_t*>(w + m.off_counters);
  float* partials = reinterpret_cast<float*>(w + m.off_partials);
  const int dpx = nseg_of(L->hidden) * 128;
  cudaError_t e;
  uint16_t* h = reinterpret_cast<uint16_t*>(w + m.off_h);
  GemvParams p = {};
  p.slots.n_slots = n_slots;
  p.slots.slot_expert = slot_expert;
  p.slots.ready = ready;
  p.slots.codes = L->gate_up_codes;
  p.slots.codes_stride = L->gate_up_codes_stride;
  p.slots.scales = L->gate_up_scales;
  p.slots.scales_stride = L->gate_up_scales_stride;
  p.slots.shared_codes = L->shared_gate_up_codes;
  p.slots.shared_scales = L->shared_gate_up_scales;
  p.slots.rows = L->inter;
  p.slots.up_row_off = L->inter;
  p.slots.tiles_per_slot = m.tiles_gu;
  p.slots.max_slots = m.max_slots;
  p.slots.n_experts = L->n_experts;
  p.N = N;
  p.d_in = L->hidden;
  p.nseg = nseg_of(L->hidden);
  p.d_in_pad = dpx;
  p.n_tiles = m.tiles_gu * m.max_slots;
  p.n_warps = gemv_max_warps();
  p.x = xp;
  p.out = h;
  p.out_ld = L->inter;
  p.out_slot_stride = (size_t)N * L->inter;
  p.counters = counters;
  p.partials = partials;
  p.partials_bytes = m.partials_bytes;
  uint32_t* status = reinterpret_cast<uint32_t*>(w + m.off_status);
  // the TMA expert kernel when the shapes allow (the caller prepared x in its
  // layout, moe_x_layout), else the first kernel
  const bool tma_gu = moe_x_layout(L, N) != 0;
  if (tma_gu && !moe_tma_eligible(kEpiSwiGLU, p)) return fail(BWS_ERR_WORKSPACE, "%s: expert kernel scratch too small", name);
  e = tma_gu ? launch_gemv_tma_moe(kEpiSwiGLU, p, status, st, true) : launch_gemv(kFmtMXFP4, kEpiSwiGLU, p, st, true);
  if (e != cudaSuccess) return cuda_status(e, name);

  char* hb = w + m.off_hp;
  PrepParams q = {};
  q.mode = kPrepCopy;
  q.x = h;
  q.ld = L->inter;
  q.x_slot_stride = (size_t)N * L->inter;
  q.N = N;
  q.d_in = L->inter;
  q.d_in_pad = nseg_of(L->inter) * 128;
  q.n_slots = n_slots;
  q.max_slots = m.max_slots;
  q.hi = reinterpret_cast<uint16_t*>(hb + m.hw.off_hi);
  q.lo = reinterpret_cast<uint16_t*>(hb + m.hw.off_lo);
  q.exp = reinterpret_cast<int*>(hb + m.hw.off_exp);
  q.flags = reinterpret_cast<uint32_t*>(hb + m.hw.off_flags);
  q.zero_ptr = counters;
  q.zero_words = m.n_tiles;
  GemvParams d = p;
  d.slots.codes = L->down_codes;
  d.slots.codes_stride = L->down_codes_stride;
  d.slots.scales = L->down_scales;
  d.slots.scales_stride = L->down_scales_stride;
  d.slots.shared_codes = L->shared_down_codes;
  d.slots.shared_scales = L->shared_down_scales;
  d.slots.rows = L->hidden;
  d.slots.up_row_off = 0;
  d.slots.tiles_per_slot = m.tiles_dn;
  d.d_in = L->inter;
  d.nseg = nseg_of(L->inter);
  d.d_in_pad = q.d_in_pad;
  d.n_tiles = m.tiles_dn * m.max_slots;
  d.x.hi = q.hi;
  d.x.lo = q.lo;
  d.x.exp = q.exp;
  d.x.flags = q.flags;
  d.x.shared = 0;
  d.out = reinterpret_cast<float*>(w + m.off_ys);
  d.out_ld = L->hidden;
  d.out_slot_stride = (size_t)N * L->hidden;
  const bool tma_dn = moe_tma_eligible(kEpiStoreF32, d);
  q.interleave = tma_dn ? 256 : 0;
  e = launch_prep(q, st, true);
  if (e != cudaSuccess) return cuda_status(e, name);
  e = tma_dn ? launch_gemv_tma_moe(kEpiStoreF32, d, status, st, true) : launch_gemv(kFmtMXFP4, kEpiStoreF32, d, st, true);
  return cuda_status(e, name);

}

// Enqueues the six kernels. out_mode: kEpiStoreBF16 (y bf16) or kEpiResidF32
// (y fp32 accumulated into). x_prepped: activations already prepared in the
// workspace's x block by the caller (the decode stream), so prep x is skipped.
int enqueue_moe(const bws_moe_layer* L, const int32_t* ids, const float* route_w, int N, int topk,
                const uint16_t* x, void* y, int out_mode, void* ws, cudaStream_t st, const XPrep* x_prepped,
                const char* name) {
  const MoeLayout m = moe_layout(L, N, topk);
  char* w = static_cast<char*>(ws);
  int* n_slots = reinterpret_cast<int*>(w + m.off_route);
  int* slot_expert = reinterpret_cast<int*>(w + m.off_slot_expert);
  float* cw = reinterpret_cast<float*>(w + m.off_cw);
  uint32_t* counters = reinterpret_cast<uint32_t*>(w + m.off_counters);
  const int has_shared = L->shared_gate_up_codes != nullptr ? 1 : 0;

  MoeRoute r = {};
  r.ids = ids;
  r.route_w = route_w;
  r.N = N;
  r.topk = topk;
  r.n_experts = L->n_experts;
  r.has_shared = has_shared;
  r.max_slots = m.max_slots;
  r.n_slots = n_slots;
  r.slot_expert = slot_expert;
  r.cw = cw;
  r.status = reinterpret_cast<uint32_t*>(w + m.off_status);
  cudaError_t e = launch_moe_route(r, st, true);
  if (e != cudaSuccess) return cuda_status(e, name);

  XPrep xp;
  const int dpx = nseg_of(L->hidden) * 128;
  if (x_prepped != nullptr) {
    xp = *x_prepped;
  } else {
    char* xb = w + m.off_x;
    PrepParams q = {};
    q.mode = kPrepCopy;
    q.x = x;
    q.ld = L->hidden;
    q.N = N;
    q.d_in = L->hidden;
    q.d_in_pad = dpx;
    q.hi = reinterpret_cast<uint16_t*>(xb + m.xw.off_hi);
    q.lo = reinterpret_cast<uint16_t*>(xb + m.xw.off_lo);
    q.exp = reinterpret_cast<int*>(xb + m.xw.off_exp);
    q.flags = reinterpret_cast<uint32_t*>(xb + m.xw.off_flags);
    q.hdr = reinterpret_cast<uint32_t*>(xb + m.xw.off_hdr);
    q.zero_ptr = counters;
    q.zero_words = m.n_tiles;
    q.interleave = moe_x_layout(L, N);
    e = launch_prep(q, st, true);
    if (e != cudaSuccess) return cuda_status(e, name);
    xp.hi = q.hi;
    xp.lo = q.lo;
    xp.exp = q.exp;
    xp.flags = q.flags;
    xp.shared = 1;
  }

  const int rc = enqueue_moe_experts(L, N, topk, n_slots, slot_expert, xp, w, st, name);
  if (rc != BWS_OK) return rc;
  float* ys = reinterpret_cast<float*>(w + m.off_ys);
  e = launch_moe_combine(ys, cw, n_slots, N, L->hidden, y, out_mode, st, true);
  return cuda_status(e, name);
}

size_t moe_workspace_bytes(const bws_moe_layer* L, int N, int topk) { return moe_layout(L, N, topk).total; }

int moe_x_layout(const bws_moe_layer* L, int N) {
  return moe_tma_shape_ok(L->gate_up_codes, L->gate_up_codes_stride, L->shared_gate_up_codes, L->gate_up_scales,
                          L->gate_up_scales_stride, L->shared_gate_up_scales, L->hidden, N)
             ? 256
             : 0;
}

MoeStackView moe_stack_view(const bws_moe_layer* L, const int32_t* ids, const float* route_w, int N, int topk,
                            void* ws, int buffer) {
  const MoeLayout m = moe_layout(L, N, topk);
  char* w = static_cast<char*>(ws);
  MoeStackView v;
  v.route.ids = ids;
  v.route.route_w = route_w;
  v.route.N = N;
  v.route.topk = topk;
  v.route.n_experts = L->n_experts;
  v.route.has_shared = L->shared_gate_up_codes != nullptr ? 1 : 0;
  v.route.max_slots = m.max_slots;
  v.route.n_slots = reinterpret_cast<int*>(w + (buffer ? m.off_route_b : m.off_route));
  v.route.slot_expert = reinterpret_cast<int*>(w + (buffer ? m.off_slot_expert_b : m.off_slot_expert));
  v.route.cw = reinterpret_cast<float*>(w + (buffer ? m.off_cw_b : m.off_cw));
  v.route.status = reinterpret_cast<uint32_t*>(w + m.off_status);
  v.ys = reinterpret_cast<float*>(w + m.off_ys);
  v.h = reinterpret_cast<uint16_t*>(w + m.off_h);
  v.counters = reinterpret_cast<uint32_t*>(w + m.off_counters);
  v.n_counters = m.n_tiles;
  return v;
}

void moe_counter_span(const bws_moe_layer* L, int N, int topk, size_t* offset, int* words) {
  const MoeLayout m = moe_layout(L, N, topk);
  *offset = m.off_counters;
  *words = m.n_tiles;
}

int check_moe_layer(const bws_moe_layer* L, int N, int topk, const char* name) { return check_moe(L, N, topk, name); }

}  // namespace bws

using namespace bws;

extern "C" {

size_t bws_mxfp4_moe_workspace_size(const bws_moe_layer* L, int N, int topk) {
  if (check_moe(L, N, topk, "bws_mxfp4_moe_workspace_size") != BWS_OK) return 0;
  return moe_layout(L, N, topk).total;
}

int bws_mxfp4_moe_gemv(const bws_moe_layer* L, const int32_t* ids, const float* route_w, int N, int topk,
                       const uint16_t* x, uint16_t* y, void* workspace, size_t workspace_bytes, void* stream) {
  const char* name = "bws_mxfp4_moe_gemv";
  int rc = check_moe(L, N, topk, name);
  if (rc) return rc;
  if (!ids || !route_w || !x || !y) return fail(BWS_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned(x, 16) || !aligned(y, 2) || !aligned(ids, 4) || !aligned(route_w, 4))
    return fail(BWS_ERR_MISALIGNED, "%s: x 16-byte, y 2-byte, ids and route_w 4-byte alignment needed", name);
  const size_t need = moe_layout(L, N, topk).total;
  if (!workspace || workspace_bytes < need)
    return fail(BWS_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", name, need, workspace_bytes);
  if (!aligned(workspace, 256)) return fail(BWS_ERR_MISALIGNED, "%s: workspace must be 256-byte aligned", name);
  return enqueue_moe(L, ids, route_w, N, topk, x, y, kEpiStoreBF16, workspace, as_stream(stream), nullptr, name);
}

int bws_mxfp4_moe_inspect(const void* workspace, const bws_moe_layer* L, int N, int topk, int* n_slots,
                          int32_t* slot_expert, uint16_t* h, uint32_t* status, void* stream) {
  const char* name = "bws_mxfp4_moe_inspect";
  int rc = check_moe(L, N, topk, name);
  if (rc) return rc;
  if (!workspace || !n_slots || !slot_expert || !h || !status) return fail(BWS_ERR_INVALID_ARG, "%s: null pointer", name);
  const MoeLayout m = moe_layout(L, N, topk);
  const char* w = static_cast<const char*>(workspace);
  cudaStream_t st = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(n_slots, w + m.off_route, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(status, w + m.off_status, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(slot_expert, w + m.off_slot_expert, sizeof(int) * m.max_slots, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(h, w + m.off_h, 2 * (size_t)m.max_slots * N * L->inter, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return cuda_status(e, name);
}

}  // extern "C"
