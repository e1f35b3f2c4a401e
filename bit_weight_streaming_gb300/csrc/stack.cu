// C ABI of the whole decode step: a validated layer stack whose kernels are
// enqueued in order on one stream, chained with programmatic dependent launch
// (each product kernel starts pulling its weights into L2 while the kernel
// before it finishes), and recorded once as a CUDA graph.
#include <cuda_runtime.h>

#include <cstdlib>
#include <new>
#include <vector>

#include "../../include/bws.h"
#include "bws_abi_util.h"
#include "bws_internal.h"
#include "step.h"

using namespace bws;

struct bws_stack_plan {
  int N, hidden;
  float eps;
  std::vector<bws_layer> layers;
  bws_matrix head;
  // workspace layout
  size_t off_status, off_r, off_xp, off_u, off_vp, off_h, off_hp, off_moe, off_counters, off_partials, total;
  // MoE layers: one slot table per layer (n_slots, slot_expert, cw) and its
  // ready flag, cleared at the start of every step
  size_t off_routes, route_stride, off_ready;
  int n_moe;
  // MoE layers with a router: the layer's normalised input (bf16 [N][hidden])
  // and logits (fp32 [N][max_router_e]) of the layer being routed; one
  // counter per MoE layer follows the ready flags
  size_t off_rx, off_rz;
  int max_router_e;
  GemvWorkspace xw, vw, hw;    // prep-block offsets (relative to their block)
  int max_u, max_dv, max_inter, max_tiles;
  int kernels;
  // dense stacks: the persistent step kernel's program (nullptr: the kernel chain)
  StepProgram* step;
  // recorded graph
  cudaGraphExec_t exec;
  const void* key[6];
};

namespace {

int check_matrix(const bws_matrix& m, int d_in, const char* what, int layer) {
  const char* name = "bws_decode_step_plan_create";
  if (m.format != BWS_FMT_NVFP4 && m.format != BWS_FMT_MXFP4 && m.format != BWS_FMT_FP8_ROW)
    return fail(BWS_ERR_FORMAT, "%s: layer %d %s: unknown format %d", name, layer, what, m.format);
  if (m.d_in != d_in || m.d_out < 1 || m.d_in % 32)
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: layer %d %s: %d x %d (d_in %d expected, %% 32)", name, layer, what,
                m.d_out, m.d_in, d_in);
  if (!m.codes || !aligned(m.codes, 16))
    return fail(BWS_ERR_MISALIGNED, "%s: layer %d %s: codes null or not 16-byte aligned", name, layer, what);
  if (m.format != BWS_FMT_FP8_ROW && !m.scales)
    return fail(BWS_ERR_INVALID_ARG, "%s: layer %d %s: null block scales", name, layer, what);
  if (m.format != BWS_FMT_MXFP4 && !m.scale32)
    return fail(BWS_ERR_INVALID_ARG, "%s: layer %d %s: null FP32 scale", name, layer, what);
  return BWS_OK;
}

int fmt_of(const bws_matrix& m) {
  return m.format == BWS_FMT_NVFP4 ? kFmtNVFP4 : (m.format == BWS_FMT_MXFP4 ? kFmtMXFP4 : kFmtFP8);
}

GemvMat gm(const bws_matrix& m, int out_row_off, int tile_begin) {
  GemvMat g;
  g.codes = m.codes;
  g.scales = m.scales;
  g.scale32 = m.scale32;
  g.d_out = m.d_out;
  g.out_row_off = out_row_off;
  g.tile_begin = tile_begin;
  return g;
}

// Verification tap (bws_decode_step_tap): records appended in launch order,
// each on a 256-byte boundary. With a null base only the sizes are counted.
struct Tap {
  char* base;
  size_t off;
  cudaStream_t st;
  cudaError_t err;
  void* take(size_t bytes) {
    void* d = base ? base + off : nullptr;
    off += align256(bytes);
    return d;
  }
  void copy(const void* src, size_t bytes) {
    void* d = take(bytes);
    if (d && err == cudaSuccess) err = cudaMemcpyAsync(d, src, bytes, cudaMemcpyDeviceToDevice, st);
  }
  void copy_to(void* d, const void* src, size_t bytes) {
    if (d && err == cudaSuccess) err = cudaMemcpyAsync(d, src, bytes, cudaMemcpyDeviceToDevice, st);
  }
  // rows of row_bytes each, src_pitch bytes apart, packed
  void copy_rows(const void* src, size_t src_pitch, size_t row_bytes, int rows) {
    void* d = take(row_bytes * rows);
    if (d && err == cudaSuccess)
      err = cudaMemcpy2DAsync(d, row_bytes, src, src_pitch, row_bytes, rows, cudaMemcpyDeviceToDevice, st);
  }
};

struct Ctx {
  const bws_stack_plan* P;
  char* w;
  cudaStream_t st;
  Tap* tap;   // optional
};

XPrep xprep_of(const Ctx& c, size_t block, const GemvWorkspace& L) {
  XPrep x;
  x.hi = reinterpret_cast<uint16_t*>(c.w + block + L.off_hi);
  x.lo = reinterpret_cast<uint16_t*>(c.w + block + L.off_lo);
  x.exp = reinterpret_cast<int*>(c.w + block + L.off_exp);
  x.flags = reinterpret_cast<uint32_t*>(c.w + block + L.off_flags);
  x.shared = 1;
  return x;
}

// prep into a block; zeroes `zero_words` counters at zero_ptr
// comb: the previous MoE layer's combine, folded into this RMSNorm prep;
// route: this MoE layer's routing, done by one extra CTA of this prep.
// A product whose outputs only the next prep reads: run by the TMA kernel,
// its CTAs deposit raw sums and that prep finishes the rows, so no CTA of
// the product waits on a fix-up. Needs tiles that never share an 8-row chunk
// with another matrix, and a finishing prep shape for the next_d rows the
// prep reads. Returns whether p now deposits; f: the prep's fields.
bool deposit_setup(const bws_matrix* mats, int nm, int epi, GemvParams& p, int next_d, PrepParams& f) {
  const int fmt = fmt_of(mats[0]);
  if (fmt == kFmtMXFP4 || epi == kEpiStoreF32 || gemv_umma_eligible(fmt, p) || !gemv_tma_eligible(fmt, p) ||
      !prep_can_finish(next_d))
    return false;
  const int rows = epi == kEpiSwiGLU ? 64 : 128;
  for (int i = 0; i < nm; ++i)
    if (mats[i].d_out % rows) return false;
  const TmaGeom geo = gemv_tma_geometry(fmt, epi, p);
  if (!gemv_tma_deposit_fits(geo, p)) return false;
  p.deposit = 1;
  f.fin_partials = p.partials;
  f.fin_split = geo.split;
  f.fin_nks = geo.nks;
  f.fin_epi = epi;
  f.fin_fmt = fmt;
  f.fin_n_mats = nm;
  int tile = 0;
  for (int i = 0; i < nm; ++i) {
    f.fin_row_off[i] = p.mats[i].out_row_off;
    f.fin_tile_begin[i] = tile;
    f.fin_scale[i] = mats[i].scale32;
    tile += mats[i].d_out / rows;
  }
  f.fin_xexp = p.x.exp;
  return true;
}

cudaError_t prep(const Ctx& c, int mode, const uint16_t* x, int ld, const uint16_t* x0, int d_in, size_t block,
                 const GemvWorkspace& L, uint32_t* zero_ptr, int zero_words, int interleave = 0,
                 const MoeStackView* comb = nullptr, const MoeRoute* route = nullptr,
                 const PrepParams* fin = nullptr, uint16_t* xout = nullptr) {
  PrepParams q = {};
  if (fin != nullptr) q = *fin;   // the finishing fields
  // xout: the BF16 row formed, written out (the router's input)
  // tap: an RMSNorm prep records the BF16 row it forms, then the residual it normalised
  const bool tap_norm = c.tap != nullptr && mode == kPrepRmsNorm;
  const size_t xbytes = 2 * (size_t)c.P->N * d_in;
  uint16_t* tap_rec = tap_norm ? static_cast<uint16_t*>(c.tap->take(xbytes)) : nullptr;
  q.tap_x = xout != nullptr ? xout : tap_rec;
  q.mode = mode;
  q.x = x;
  q.ld = ld;
  q.r = reinterpret_cast<float*>(c.w + c.P->off_r);
  q.x0 = x0;
  q.eps = c.P->eps;
  q.N = c.P->N;
  q.d_in = d_in;
  q.d_in_pad = nseg_of(d_in) * 128;
  const XPrep xp = xprep_of(c, block, L);
  q.hi = const_cast<uint16_t*>(xp.hi);
  q.lo = const_cast<uint16_t*>(xp.lo);
  q.exp = const_cast<int*>(xp.exp);
  q.flags = const_cast<uint32_t*>(xp.flags);
  q.hdr = nullptr;
  q.status_clear = x0 != nullptr ? reinterpret_cast<uint32_t*>(c.w + c.P->off_status) : nullptr;   // words 0, 1
  q.zero_ptr = zero_ptr;
  q.zero_words = zero_words;
  q.interleave = interleave;
  if (comb != nullptr) {
    q.comb_ys = comb->ys;
    q.comb_cw = comb->route.cw;
    q.comb_n_slots = comb->route.n_slots;
    q.comb_max_slots = comb->route.max_slots;
    q.comb_tok_slots = comb->route.tok_slots;
    q.comb_topk = comb->route.topk;
    q.comb_has_shared = comb->route.has_shared;
  }
  if (route != nullptr) {
    q.has_route = 1;
    q.route = *route;
  }
  const cudaError_t e = launch_prep(q, c.st, true);
  if (e == cudaSuccess && tap_norm) {
    if (xout != nullptr) c.tap->copy_to(tap_rec, xout, xbytes);
    c.tap->copy(q.r, sizeof(float) * (size_t)c.P->N * d_in);
  }
  return e;
}

int tiles_for(const bws_matrix* mats, int nm, int epi) {
  if (epi == kEpiSwiGLU) return (mats[0].d_out + 15) / 16;
  int t = 0;
  for (int i = 0; i < nm; ++i) t += (mats[i].d_out + 31) / 32;
  return t;
}

GemvParams product_params(const Ctx& c, const bws_matrix* mats, int nm, int epi, int d_in, const XPrep& x,
                          void* out, int out_ld) {
  GemvParams p = {};
  p.n_mats = nm;
  int tile = 0, row = 0;
  for (int i = 0; i < nm; ++i) {
    p.mats[i] = gm(mats[i], epi == kEpiSwiGLU ? 0 : row, tile);
    row += mats[i].d_out;
    tile += (mats[i].d_out + 31) / 32;
  }
  p.n_tiles = tiles_for(mats, nm, epi);
  p.N = c.P->N;
  p.d_in = d_in;
  p.nseg = nseg_of(d_in);
  p.d_in_pad = p.nseg * 128;
  p.n_units = (long long)p.n_tiles * p.nseg;
  const long long maxw = gemv_max_warps();
  p.n_warps = p.n_units < maxw ? p.n_units : maxw;
  p.x = x;
  p.out = out;
  p.out_ld = out_ld;
  p.counters = reinterpret_cast<uint32_t*>(c.w + c.P->off_counters);
  p.partials = reinterpret_cast<float*>(c.w + c.P->off_partials);
  p.prefetch_units = fmt_of(mats[0]) == kFmtFP8 ? 4 : 8;
  return p;
}

// The activation layout the product's kernel reads.
int layout_for(const bws_matrix* mats, const GemvParams& p) {
  const int fmt = fmt_of(mats[0]);
  return product_layout(fmt, p);
}

cudaError_t product(const Ctx& c, const bws_matrix* mats, int nm, int epi, const GemvParams& p) {
  return launch_product(fmt_of(mats[0]), epi, p, reinterpret_cast<uint32_t*>(c.w + c.P->off_status) + 1, c.st,
                        true);
}

int enqueue_step(const bws_stack_plan* P, const uint16_t* x0, float* logits, const int32_t* row_token,
                 int32_t* tokens, void* ws, cudaStream_t st, Tap* tap = nullptr) {
  const char* name = tap ? "bws_decode_step_tap" : (tokens ? "bws_decode_step_greedy" : "bws_decode_step_stream");
  if (P->step) {
    if (tap || tokens)
      return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: the persistent step kernel has no tap or fused argmax", name);
    return cuda_status(step_program_enqueue(P->step, x0, logits, ws, st), name);
  }
  Ctx c{P, static_cast<char*>(ws), st, tap};
  float* r = reinterpret_cast<float*>(c.w + P->off_r);
  uint32_t* counters = reinterpret_cast<uint32_t*>(c.w + P->off_counters);
  uint16_t* u = reinterpret_cast<uint16_t*>(c.w + P->off_u);
  uint16_t* h = reinterpret_cast<uint16_t*>(c.w + P->off_h);
  const XPrep xa = xprep_of(c, P->off_xp, P->xw);
  const XPrep xv = xprep_of(c, P->off_vp, P->vw);
  const XPrep xh = xprep_of(c, P->off_hp, P->hw);
  const int H = P->hidden;
  const uint16_t* init = x0;   // the first RMSNorm also sets r = x0
  // an MoE layer's combine is folded into the next RMSNorm prep; its route
  // buffers alternate between consecutive MoE layers
  MoeStackView pend_v;
  const MoeStackView* pending = nullptr;
  int moe_buf = 0, moe_i = 0;
  if (P->n_moe > 0) {
    const cudaError_t e0 = cudaMemsetAsync(c.w + P->off_ready, 0, 2 * sizeof(uint32_t) * (size_t)P->n_moe, st);
    if (e0 != cudaSuccess) return cuda_status(e0, name);
  }
  // the last product's rows, when it deposited them for the next prep
  PrepParams fin_v = {};
  const PrepParams* fin = nullptr;
  // the product's CTAs that start late: the slots the prep before it (of rows
  // of d values, finishing when fin is set) holds, on about twice as many
  auto late_ctas = [&](int d) { return 2 * prep_ctas_per_row(d, fin != nullptr); };
  auto deposit = [&](const bws_matrix* mats, int nm, int epi, GemvParams& p, int next_d) {
    fin_v = PrepParams{};
    fin = deposit_setup(mats, nm, epi, p, next_d, fin_v) ? &fin_v : nullptr;
  };
  cudaError_t e = cudaSuccess;
#define BWS_TRY(call)                          \
  do {                                         \
    e = (call);                                \
    if (e != cudaSuccess) return cuda_status(e, name); \
  } while (0)
  for (size_t li = 0; li < P->layers.size(); ++li) {
    const bws_layer& L = P->layers[li];
    if (L.kind == BWS_LAYER_MIXER_MLP) {
      int sum_out = 0;
      for (int i = 0; i < L.n_mixer_in; ++i) sum_out += L.mixer_in[i].d_out;
      GemvParams pin = product_params(c, L.mixer_in, L.n_mixer_in, kEpiStoreBF16, H, xa, u, sum_out);
      pin.split_light = late_ctas(H);
      BWS_TRY(prep(c, kPrepRmsNorm, nullptr, 0, init, H, P->off_xp, P->xw, counters,
                   tiles_for(L.mixer_in, L.n_mixer_in, kEpiStoreBF16), layout_for(L.mixer_in, pin), pending,
                   nullptr, fin));
      init = nullptr;
      pending = nullptr;
      deposit(L.mixer_in, L.n_mixer_in, kEpiStoreBF16, pin, L.mixer_out.d_in);
      BWS_TRY(product(c, L.mixer_in, L.n_mixer_in, kEpiStoreBF16, pin));
      const int dv = L.mixer_out.d_in;
      GemvParams pout = product_params(c, &L.mixer_out, 1, kEpiResidF32, dv, xv, r, H);
      pout.split_light = late_ctas(dv);
      BWS_TRY(prep(c, kPrepCopy, u, sum_out, nullptr, dv, P->off_vp, P->vw, counters,
                   tiles_for(&L.mixer_out, 1, kEpiResidF32), layout_for(&L.mixer_out, pout), nullptr, nullptr, fin));
      if (tap) tap->copy_rows(u, 2 * (size_t)sum_out, 2 * (size_t)dv, P->N);
      deposit(&L.mixer_out, 1, kEpiResidF32, pout, H);
      BWS_TRY(product(c, &L.mixer_out, 1, kEpiResidF32, pout));
    }
    if (L.kind == BWS_LAYER_MIXER_MLP || L.kind == BWS_LAYER_MLP) {
      const bws_matrix gu[2] = {L.gate, L.up};
      GemvParams pgu = product_params(c, gu, 2, kEpiSwiGLU, H, xa, h, L.gate.d_out);
      pgu.split_light = late_ctas(H);
      BWS_TRY(prep(c, kPrepRmsNorm, nullptr, 0, init, H, P->off_xp, P->xw, counters, tiles_for(gu, 2, kEpiSwiGLU),
                   layout_for(gu, pgu), pending, nullptr, fin));
      init = nullptr;
      pending = nullptr;
      deposit(gu, 2, kEpiSwiGLU, pgu, L.gate.d_out);
      BWS_TRY(product(c, gu, 2, kEpiSwiGLU, pgu));
      const int I = L.down.d_in;
      GemvParams pdn = product_params(c, &L.down, 1, kEpiResidF32, I, xh, r, H);
      pdn.split_light = late_ctas(I);
      BWS_TRY(prep(c, kPrepCopy, h, I, nullptr, I, P->off_hp, P->hw, counters, tiles_for(&L.down, 1, kEpiResidF32),
                   layout_for(&L.down, pdn), nullptr, nullptr, fin));
      if (tap) tap->copy(h, 2 * (size_t)P->N * I);
      // the next prep finishes the down rows unless it is an MoE layer's
      // (routing and combine), which reads r as the product leaves it
      const bool next_moe = li + 1 < P->layers.size() && P->layers[li + 1].kind == BWS_LAYER_MOE;
      if (next_moe)
        fin = nullptr;
      else
        deposit(&L.down, 1, kEpiResidF32, pdn, H);
      BWS_TRY(product(c, &L.down, 1, kEpiResidF32, pdn));
    }
    if (L.kind == BWS_LAYER_MOE) {
      MoeStackView v = moe_stack_view(&L.moe, L.ids, L.route_w, P->N, L.topk, c.w + P->off_moe, moe_buf);
      {   // this layer's own table, routed ahead of the layer (MoeRoute::ready)
        char* rt = c.w + P->off_routes + (size_t)moe_i * P->route_stride;
        v.route.n_slots = reinterpret_cast<int*>(rt);
        v.route.slot_expert = reinterpret_cast<int*>(rt + 256);
        v.route.cw = reinterpret_cast<float*>(rt + 256 + align256(sizeof(int) * (size_t)v.route.max_slots));
        v.route.tok_slots = reinterpret_cast<int*>(reinterpret_cast<char*>(v.route.cw) +
                                                   align256(sizeof(float) * (size_t)v.route.max_slots * P->N));
        v.route.ready = reinterpret_cast<uint32_t*>(c.w + P->off_ready) + moe_i;
      }
      if (L.router == nullptr) {   // ids known before the layer: routed by an extra CTA of the prep
        BWS_TRY(prep(c, kPrepRmsNorm, nullptr, 0, init, H, P->off_xp, P->xw, v.counters, v.n_counters,
                     moe_x_layout(&L.moe, P->N), pending, &v.route));
      } else {   // the router reads the prep's BF16 row, then writes ids, weights and the slot table
        uint16_t* rx = reinterpret_cast<uint16_t*>(c.w + P->off_rx);
        BWS_TRY(prep(c, kPrepRmsNorm, nullptr, 0, init, H, P->off_xp, P->xw, v.counters, v.n_counters,
                     moe_x_layout(&L.moe, P->N), pending, nullptr, nullptr, rx));
        RouterParams rp = {};
        rp.W = L.router;
        rp.x = rx;
        rp.N = P->N;
        rp.E = L.moe.n_experts;
        rp.d = H;
        rp.topk = L.topk;
        rp.z = reinterpret_cast<float*>(c.w + P->off_rz);
        rp.counter = reinterpret_cast<uint32_t*>(c.w + P->off_ready) + P->n_moe + moe_i;
        rp.ids = const_cast<int32_t*>(L.ids);
        rp.route_w = const_cast<float*>(L.route_w);
        rp.has_route = 1;
        rp.route = v.route;
        BWS_TRY(launch_router(rp, st, true));
        if (tap) {
          tap->copy(rp.z, sizeof(float) * (size_t)P->N * rp.E);
          tap->copy(L.ids, sizeof(int32_t) * (size_t)P->N * L.topk);
          tap->copy(L.route_w, sizeof(float) * (size_t)P->N * L.topk);
        }
      }
      ++moe_i;
      init = nullptr;
      const int rc = enqueue_moe_experts(&L.moe, P->N, L.topk, v.route.n_slots, v.route.slot_expert, xa,
                                         c.w + P->off_moe, st, name, v.route.ready);
      if (rc != BWS_OK) return rc;
      if (tap) {
        const int ms = v.route.max_slots;
        tap->copy(v.route.n_slots, sizeof(int));
        tap->copy(v.route.slot_expert, sizeof(int) * (size_t)ms);
        tap->copy(v.route.cw, sizeof(float) * (size_t)ms * P->N);
        tap->copy(v.h, 2 * (size_t)ms * P->N * L.moe.inter);
        tap->copy(v.ys, sizeof(float) * (size_t)ms * P->N * H);
      }
      pend_v = v;
      pending = &pend_v;
      moe_buf ^= 1;
    }
  }
  GemvParams ph = product_params(c, &P->head, 1, kEpiStoreF32, H, xa, logits, P->head.d_out);
  ph.split_light = late_ctas(H);
  const int head_tiles = tiles_for(&P->head, 1, kEpiStoreF32);
  int head_zero = head_tiles;
  if (tokens != nullptr) {   // greedy argmax fused into the output layer: keys after its tile counters
    if (!gemv_tma_eligible(fmt_of(P->head), ph) || gemv_umma_eligible(fmt_of(P->head), ph))
      return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: the fused argmax needs the TMA output-layer kernel", name);
    ph.amax_key = reinterpret_cast<unsigned long long*>(counters + argmax_key_word(head_tiles));
    ph.no_store = logits == nullptr;
    head_zero = argmax_key_word(head_tiles) + 2 * P->N;
  }
  BWS_TRY(prep(c, kPrepRmsNorm, nullptr, 0, init, H, P->off_xp, P->xw, counters, head_zero,
               layout_for(&P->head, ph), pending, nullptr, fin));
  BWS_TRY(product(c, &P->head, 1, kEpiStoreF32, ph));
  if (tokens != nullptr) BWS_TRY(launch_argmax_finish(ph.amax_key, P->N, row_token, tokens, st, true));
#undef BWS_TRY
  return BWS_OK;
}

// The tap's record sizes, in the order enqueue_step writes them.
size_t tap_walk_size(const bws_stack_plan* P, Tap* t) {
  const size_t N = P->N, H = P->hidden;
  for (const bws_layer& L : P->layers) {
    if (L.kind == BWS_LAYER_MIXER_MLP) {
      t->take(2 * N * H);                            // a = BF16(RMSNorm(r))
      t->take(4 * N * H);                            // the r it normalised
      t->take(2 * N * (size_t)L.mixer_out.d_in);     // v = the mixer inputs' first d_v outputs
    }
    if (L.kind == BWS_LAYER_MIXER_MLP || L.kind == BWS_LAYER_MLP) {
      t->take(2 * N * H);                            // m
      t->take(4 * N * H);                            // the r it normalised
      t->take(2 * N * (size_t)L.gate.d_out);         // h
    }
    if (L.kind == BWS_LAYER_MOE) {
      const size_t ms = N * L.topk + (L.moe.shared_gate_up_codes != nullptr ? 1 : 0);
      t->take(2 * N * H);                            // m
      t->take(4 * N * H);                            // the r it normalised
      if (L.router != nullptr) {
        t->take(4 * N * (size_t)L.moe.n_experts);    // router logits
        t->take(4 * N * (size_t)L.topk);             // chosen ids
        t->take(4 * N * (size_t)L.topk);             // their weights
      }
      t->take(sizeof(int));                          // live slots
      t->take(sizeof(int) * ms);                     // slot experts
      t->take(sizeof(float) * ms * N);               // combine weights
      t->take(2 * ms * N * L.moe.inter);             // h per slot
      t->take(sizeof(float) * ms * N * H);           // y per slot
    }
  }
  t->take(2 * N * H);                                // the output layer's input
  t->take(4 * N * H);                                // the r it normalised
  return t->off;
}

}  // namespace

extern "C" {

int bws_decode_step_plan_create(const bws_stack* S, int N, bws_stack_plan** plan) {
  const char* name = "bws_decode_step_plan_create";
  if (!S || !plan) return fail(BWS_ERR_INVALID_ARG, "%s: null pointer", name);
  *plan = nullptr;
  if (N < 1 || N > kMaxTokens) return fail(BWS_ERR_INVALID_ARG, "%s: N = %d must be in [1, %d]", name, N, kMaxTokens);
  if (S->hidden < 32 || S->hidden % 32) return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: hidden %% 32 != 0", name);
  if (S->n_layers < 0 || (S->n_layers > 0 && !S->layers)) return fail(BWS_ERR_INVALID_ARG, "%s: bad layer array", name);
  if (!(S->rms_eps >= 0.0f)) return fail(BWS_ERR_INVALID_ARG, "%s: rms_eps must be >= 0", name);
  const int H = S->hidden;
  int rc;
  bws_stack_plan* P = new (std::nothrow) bws_stack_plan();
  if (!P) return fail(BWS_ERR_INVALID_ARG, "%s: out of host memory", name);
  P->N = N;
  P->hidden = H;
  P->eps = S->rms_eps;
  P->head = S->head;
  P->max_u = P->max_dv = P->max_inter = 32;
  P->max_tiles = 1;
  P->kernels = 2;
  size_t moe_bytes = 0, route_bytes = 256;
  P->n_moe = 0;
  P->max_router_e = 0;
  auto bad = [&](int code) {
    delete P;
    return code;
  };
  for (int li = 0; li < S->n_layers; ++li) {
    const bws_layer& L = S->layers[li];
    if (L.kind == BWS_LAYER_MIXER_MLP) {
      if (L.n_mixer_in < 1 || L.n_mixer_in > 4)
        return bad(fail(BWS_ERR_INVALID_ARG, "%s: layer %d: n_mixer_in must be 1..4", name, li));
      int sum_out = 0, tiles = 0;
      for (int i = 0; i < L.n_mixer_in; ++i) {
        if ((rc = check_matrix(L.mixer_in[i], H, "mixer_in", li))) return bad(rc);
        if (L.mixer_in[i].format != L.mixer_in[0].format)
          return bad(fail(BWS_ERR_FORMAT, "%s: layer %d: mixer inputs must share one format", name, li));
        sum_out += L.mixer_in[i].d_out;
        tiles += (L.mixer_in[i].d_out + 31) / 32;
      }
      if ((rc = check_matrix(L.mixer_out, L.mixer_out.d_in, "mixer_out", li))) return bad(rc);
      if (L.mixer_out.d_out != H || L.mixer_out.d_in > sum_out)
        return bad(fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: layer %d: mixer_out must be [hidden][d_v], d_v <= %d", name, li, sum_out));
      if (sum_out % 8) return bad(fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: layer %d: mixer outputs %% 8 != 0", name, li));
      P->max_u = sum_out > P->max_u ? sum_out : P->max_u;
      P->max_dv = L.mixer_out.d_in > P->max_dv ? L.mixer_out.d_in : P->max_dv;
      P->max_tiles = tiles > P->max_tiles ? tiles : P->max_tiles;
      const int t2 = (H + 31) / 32;
      P->max_tiles = t2 > P->max_tiles ? t2 : P->max_tiles;
      P->kernels += 4;
    }
    if (L.kind == BWS_LAYER_MIXER_MLP || L.kind == BWS_LAYER_MLP) {
      if ((rc = check_matrix(L.gate, H, "gate", li)) || (rc = check_matrix(L.up, H, "up", li))) return bad(rc);
      if ((rc = check_matrix(L.down, L.gate.d_out, "down", li))) return bad(rc);
      if (L.up.d_out != L.gate.d_out || L.up.format != L.gate.format || L.down.d_out != H)
        return bad(fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: layer %d: gate/up/down shapes or formats disagree", name, li));
      const int I = L.gate.d_out;
      P->max_inter = I > P->max_inter ? I : P->max_inter;
      const int t1 = (I + 15) / 16, t2 = (H + 31) / 32;
      P->max_tiles = t1 > P->max_tiles ? t1 : P->max_tiles;
      P->max_tiles = t2 > P->max_tiles ? t2 : P->max_tiles;
      P->kernels += 4;
    } else if (L.kind == BWS_LAYER_MOE) {
      if ((rc = check_moe_layer(&L.moe, N, L.topk, name))) return bad(rc);
      if (L.moe.hidden != H) return bad(fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: layer %d: MoE hidden != stack hidden", name, li));
      if (!L.ids || !L.route_w) return bad(fail(BWS_ERR_INVALID_ARG, "%s: layer %d: null routing", name, li));
      if (L.router != nullptr) {
        if (!aligned(L.router, 16) || !aligned(L.ids, 4) || !aligned(L.route_w, 4))
          return bad(fail(BWS_ERR_MISALIGNED, "%s: layer %d: router 16-byte, ids and route_w 4-byte alignment needed",
                          name, li));
        if (L.moe.n_experts > kRouterMaxExperts || H % 8 || H > kRouterMaxD || L.topk > L.moe.n_experts)
          return bad(fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: layer %d: router needs n_experts <= %d, hidden %% 8 == 0, "
                          "hidden <= %d, topk <= n_experts", name, li, kRouterMaxExperts, kRouterMaxD));
        P->max_router_e = L.moe.n_experts > P->max_router_e ? L.moe.n_experts : P->max_router_e;
        ++P->kernels;
      }
      const size_t b = moe_workspace_bytes(&L.moe, N, L.topk);
      moe_bytes = b > moe_bytes ? b : moe_bytes;
      const size_t slots = (size_t)N * L.topk + (L.moe.shared_gate_up_codes != nullptr ? 1 : 0);
      const size_t rb = 256 + align256(sizeof(int) * slots) + align256(sizeof(float) * slots * N) +
                        align256(sizeof(int) * (size_t)N * L.topk);
      route_bytes = rb > route_bytes ? rb : route_bytes;
      ++P->n_moe;
      P->kernels += 4;
    } else if (L.kind != BWS_LAYER_MIXER_MLP) {
      return bad(fail(BWS_ERR_INVALID_ARG, "%s: layer %d: unknown kind %d", name, li, L.kind));
    }
    P->layers.push_back(L);
  }
  if ((rc = check_matrix(S->head, H, "head", -1))) return bad(rc);
  const int th = argmax_key_word((S->head.d_out + 31) / 32) + 2 * kMaxTokens;   // tile counters, argmax keys
  P->max_tiles = th > P->max_tiles ? th : P->max_tiles;
  // workspace layout
  size_t o = 0;
  P->off_status = o; o += 256;
  P->off_r = o; o += align256(sizeof(float) * (size_t)N * H);
  P->xw = gemv_workspace_layout(N, H, 0, 0, 1);
  P->off_xp = o; o += P->xw.off_counters;
  P->off_u = o; o += align256(2 * (size_t)N * P->max_u);
  P->vw = gemv_workspace_layout(N, P->max_dv, 0, 0, 1);
  P->off_vp = o; o += P->vw.off_counters;
  P->off_h = o; o += align256(2 * (size_t)N * P->max_inter);
  P->hw = gemv_workspace_layout(N, P->max_inter, 0, 0, 1);
  P->off_hp = o; o += P->hw.off_counters;
  P->off_moe = o; o += align256(moe_bytes);
  P->route_stride = route_bytes;
  P->off_routes = o; o += route_bytes * (size_t)P->n_moe;
  P->off_ready = o; o += align256(2 * sizeof(uint32_t) * (size_t)(P->n_moe > 0 ? P->n_moe : 1));
  P->off_rx = o; o += P->max_router_e > 0 ? align256(2 * (size_t)N * H) : 0;
  P->off_rz = o; o += align256(sizeof(float) * (size_t)N * P->max_router_e);
  P->off_counters = o; o += align256(sizeof(uint32_t) * (size_t)P->max_tiles);
  P->off_partials = o; o += align256(sizeof(float) * kSlotFloats * ((size_t)P->max_tiles + gemv_max_warps()));
  P->total = o;
  // A dense stack can run as one persistent kernel. It is opt-in
  // (BWS_STEP_KERNEL=1 at plan creation) until it outruns the kernel chain.
  const char* opt = getenv("BWS_STEP_KERNEL");
  P->step = (opt && opt[0] == '1')
                ? step_program_create(N, H, P->eps, P->layers.data(), (int)P->layers.size(), P->head)
                : nullptr;
  if (P->step) {   // the chain's buffers are not used
    P->total = step_program_workspace(P->step);
    P->kernels = 2;
  }
  P->exec = nullptr;
  for (auto& k : P->key) k = nullptr;
  *plan = P;
  clear_error();
  return BWS_OK;
}

void bws_decode_step_plan_destroy(bws_stack_plan* plan) {
  if (!plan) return;
  if (plan->exec) cudaGraphExecDestroy(plan->exec);
  step_program_destroy(plan->step);
  delete plan;
}

size_t bws_decode_step_workspace_size(const bws_stack_plan* plan) { return plan ? plan->total : 0; }

int bws_decode_step_kernel_count(const bws_stack_plan* plan) { return plan ? plan->kernels : 0; }

size_t bws_decode_step_tap_size(const bws_stack_plan* plan) {
  if (!plan || plan->step) return 0;
  Tap t{nullptr, 0, nullptr, cudaSuccess};
  return tap_walk_size(plan, &t);
}

int bws_decode_step_tap(bws_stack_plan* P, const uint16_t* x0, float* logits, void* ws, size_t ws_bytes, void* tap,
                        size_t tap_bytes, void* stream) {
  const char* name = "bws_decode_step_tap";
  if (!P || !x0 || !logits || !ws || !tap) return fail(BWS_ERR_INVALID_ARG, "%s: null pointer", name);
  if (P->step) return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: the persistent step kernel has no tap", name);
  if (ws_bytes < P->total) return fail(BWS_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", name, P->total, ws_bytes);
  const size_t need = bws_decode_step_tap_size(P);
  if (tap_bytes < need) return fail(BWS_ERR_WORKSPACE, "%s: tap of %zu bytes needed, %zu given", name, need, tap_bytes);
  if (!aligned(ws, 256) || !aligned(tap, 256) || !aligned(x0, 16) || !aligned(logits, 4))
    return fail(BWS_ERR_MISALIGNED, "%s: workspace and tap 256-byte, x0 16-byte, logits 4-byte alignment needed", name);
  cudaStream_t st = as_stream(stream);
  Tap t{static_cast<char*>(tap), 0, st, cudaSuccess};
  const int rc = enqueue_step(P, x0, logits, nullptr, nullptr, ws, st, &t);
  if (rc != BWS_OK) return rc;
  return cuda_status(t.err, name);
}

static int run_step(bws_stack_plan* P, const uint16_t* x0, float* logits, const int32_t* row_token, int32_t* tokens,
                    void* ws, size_t ws_bytes, void* stream, const char* name) {
  if (!P || !x0 || !ws || (!logits && !tokens)) return fail(BWS_ERR_INVALID_ARG, "%s: null pointer", name);
  if (ws_bytes < P->total) return fail(BWS_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", name, P->total, ws_bytes);
  if (!aligned(ws, 256) || !aligned(x0, 16) || !aligned(logits, 4) || !aligned(tokens, 4) || !aligned(row_token, 4))
    return fail(BWS_ERR_MISALIGNED, "%s: workspace 256-byte, x0 16-byte, logits and tokens 4-byte alignment needed", name);
  cudaStream_t st = as_stream(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (st != nullptr) {
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return cuda_status(e, name);
  }
  if (st == nullptr || cs != cudaStreamCaptureStatusNone) return enqueue_step(P, x0, logits, row_token, tokens, ws, st);
  const void* key[6] = {x0, logits, ws, st, row_token, tokens};
  bool same = P->exec != nullptr;
  for (int i = 0; i < 6; ++i) same = same && key[i] == P->key[i];
  if (!same) {
    if (P->exec) {
      cudaGraphExecDestroy(P->exec);
      P->exec = nullptr;
    }
    cudaError_t e = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_status(e, name);
    const int rc = enqueue_step(P, x0, logits, row_token, tokens, ws, st);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(st, &g);
    if (rc != BWS_OK) {
      if (g) cudaGraphDestroy(g);
      return rc;
    }
    if (e != cudaSuccess) return cuda_status(e, name);
    e = cudaGraphInstantiate(&P->exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      P->exec = nullptr;
      return cuda_status(e, name);
    }
    for (int i = 0; i < 6; ++i) P->key[i] = key[i];
  }
  return cuda_status(cudaGraphLaunch(P->exec, st), name);
}

int bws_decode_step_stream(bws_stack_plan* P, const uint16_t* x0, float* logits, void* ws, size_t ws_bytes,
                           void* stream) {
  if (!logits) return fail(BWS_ERR_INVALID_ARG, "bws_decode_step_stream: null logits");
  return run_step(P, x0, logits, nullptr, nullptr, ws, ws_bytes, stream, "bws_decode_step_stream");
}

int bws_decode_step_greedy(bws_stack_plan* P, const uint16_t* x0, float* logits, const int32_t* row_token,
                           int32_t* tokens, void* ws, size_t ws_bytes, void* stream) {
  if (!tokens) return fail(BWS_ERR_INVALID_ARG, "bws_decode_step_greedy: null tokens");
  return run_step(P, x0, logits, row_token, tokens, ws, ws_bytes, stream, "bws_decode_step_greedy");
}

}  // extern "C"
