// One decode step over every layer, pipelined as InfiniGen's KV selection controller and
// inference controller are (paper-graph summary, section 3.2 architecture and section 3.4,
// "Decoding Stage", Step 5 and Fig 8): while layer i-1 computes, layer i is speculated from
// layer i-1's input and its selected rows are fetched on a side stream; layer 0 attends over
// its full, HBM-resident KV.
//
// Per step, on the compute stream S and the fetch stream G:
//   for l = 1 .. L-1:
//     S: speculate(l) from layer l-1's input, select(l), record sel[l]
//     G: wait sel[l] (and att[l-2], which frees gather buffer l % 2), gather(l), record got[l]
//     S: (l >= 2: wait got[l-1]) attention(l-1), append(l-1), record att[l-1]
//        (attention(0) is the dense layer-0 attention, which needs no fetch)
//   S: wait got[L-1], attention(L-1), append(L-1)
// so layer 1 is speculated and its fetch starts before layer 0 attends.
//
// With config.fused_fetch the selected rows are not staged in HBM: the fetch stream reads them
// from the pinned pool and folds them into per-head partial attention (the partials of
// ig_gather_attend), and the compute stream merges them (its combine):
//   for l = 1 .. L-1:
//     S: (l >= 3: wait att[l-2]; combine(l-2), the attention that yields layer l-1's input;
//        append(l-2))
//        speculate(l), select(l), record sel[l]
//     G: wait sel[l], fetch + partial attention(l) into partial set l % 2, record att[l]
//     S: (l == 1) dense attention(0), append(0)
//   S: wait att[L-2], combine + append(L-2); wait att[L-1], combine + append(L-1)
// so the fetch stream does nothing but fetch and attend.  Selection l reuses index buffer
// l % 2, and the fetch of layer l partial set l % 2, only after combine(l-2) (which S runs
// before selection l) is done with them (config.keep_indices gives every layer an index list
// of its own instead).
#include <limits>
#include <vector>

#include "ig_common.cuh"
#include "pool_impl.h"

namespace ig {
ig_status fetch_attend_partials(cudaStream_t s, const ig_pool* pool, int layer, int B, int H, int d, int Lcap,
                                float scale, const uint16_t* q, const int32_t* idx, const int32_t* cnt,
                                const uint16_t* k_new, const uint16_t* v_new, const float* out, void* workspace,
                                size_t workspace_bytes, int max_ctas, int* grid_out);
ig_status fetch_attend_combine(cudaStream_t s, int B, int H, int d, float scale, const uint16_t* q,
                               const uint16_t* k_new, const uint16_t* v_new, float* out, const void* workspace,
                               int grid);
}  // namespace ig

struct ig_decoder {
  ig_decoder_config cfg{};
  ig_decoder_buffers buf{};
  std::vector<const uint16_t*> Wq_part, Wq;
  std::vector<const float*> A_cols;
  std::vector<uint16_t*> Kpart;
  std::vector<const int32_t*> cols;
  std::vector<int> ks;  // partial width of each layer (config k when none is given)
  ig_pool* pool = nullptr;
  std::vector<cudaEvent_t> ev_sel, ev_got, ev_att;
  size_t ws_main = 0, ws_sel = 0, ws_fetch = 0;  // workspace regions: S, selection, G (fused fetch)
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // stage timing (optional): start/end of gather (G), speculate+select and attention+append
  // (S); two sets, alternating by step, indexed [parity * layers + layer]
  std::vector<cudaEvent_t> tg0, tg1, ts0, ts1, ta0, ta1;
  long long steps = 0;  // decode steps enqueued so far
  // captured steps (ig_decoder_graph_capture), one per timing-event set
  cudaGraphExec_t graph[2] = {nullptr, nullptr};
  uint64_t graph_kernels = 0;  // kernels in one captured step
};

namespace {

size_t sz_scores(const ig_decoder_config& c) { return (size_t)c.B * c.H * c.Lcap; }
size_t sz_kv(const ig_decoder_config& c) { return (size_t)c.B * c.H * c.Lcap * c.d; }
// offset of layer l's index list: one list per layer, or two reused by layer parity
size_t idx_off(const ig_decoder_config& c, int l) {
  return (size_t)(c.keep_indices ? l : (l & 1)) * sz_scores(c);
}

void destroy_events(ig_decoder* d) {
  for (auto* v : {&d->ev_sel, &d->ev_got, &d->ev_att, &d->tg0, &d->tg1, &d->ts0, &d->ts1, &d->ta0,
                  &d->ta1})
    for (cudaEvent_t e : *v)
      if (e) cudaEventDestroy(e);
  if (d->ev_fork) cudaEventDestroy(d->ev_fork);
  if (d->ev_join) cudaEventDestroy(d->ev_join);
  for (cudaGraphExec_t& g : d->graph)
    if (g) {
      cudaGraphExecDestroy(g);
      g = nullptr;
    }
}

}  // namespace

using namespace ig;

namespace {

// workspace regions: [main: speculation / selection-fused / S's attention][selection][fetch
// stream's attention, fused fetch only]
void ws_regions(const ig_decoder_config* c, size_t* main, size_t* sel, size_t* fetch) {
  const bool rope = c->rope_theta > 0.f;
  size_t a = rope ? ig_speculate_rope_workspace_bytes(c->B, c->D, c->H, c->d, c->k)
                  : ig_speculate_workspace_bytes(c->B, c->D, c->H, c->k);
  const size_t f = ig_speculate_select_workspace_bytes(c->B, c->D, c->H, c->d, c->k, rope ? 1 : 0);
  if (f > a) a = f;
  const size_t b = ig_attend_workspace_bytes(c->B, c->H, c->d, c->Lcap);
  *main = round_up(a > b ? a : b, 256);
  *sel = round_up(ig_select_workspace_bytes(c->B, c->H), 256);
  // fused fetch: two partial sets, by layer parity (the combine of layer l runs on the compute
  // stream while the fetch stream writes layer l+1's partials)
  *fetch = c->fused_fetch ? 2 * round_up(ig_gather_attend_workspace_bytes(c->B, c->H, c->d, c->Lcap), 256) : 0;
}

}  // namespace

extern "C" size_t ig_decoder_workspace_bytes(const ig_decoder_config* c) {
  if (!c) return 0;
  size_t m, s, f;
  ws_regions(c, &m, &s, &f);
  return m + s + f;
}

extern "C" ig_status ig_decoder_create(const ig_decoder_config* cfg, const ig_decoder_buffers* buf,
                                       ig_pool* pool, ig_decoder** out) {
  IG_REQUIRE(cfg && buf && out, "null argument");
  *out = nullptr;
  const ig_decoder_config& c = *cfg;
  IG_REQUIRE(c.layers >= 1 && c.B > 0 && c.H > 0 && c.d > 0 && c.D > 0 && c.k > 0 && c.k <= c.d,
             "bad decoder sizes");
  IG_REQUIRE(c.Lcap > 0 && c.Lcap % 8 == 0, "Lcap must be a positive multiple of 8");
  IG_REQUIRE(c.alpha > 0.f, "alpha must be > 0");
  IG_REQUIRE(pool && pool->layers == c.layers && pool->B == c.B && pool->H == c.H && pool->d == c.d,
             "pool does not match the decoder");
  IG_REQUIRE(pool->cap <= c.Lcap, "pool capacity %d exceeds Lcap %d", pool->cap, c.Lcap);
  IG_REQUIRE(buf->Kpart && buf->cols && buf->K0 && buf->V0 && buf->scores && buf->idx && buf->cnt &&
                 buf->workspace,
             "missing decoder buffer");
  IG_REQUIRE(c.fused_fetch || (buf->Kg && buf->Vg), "staged fetch needs Kg and Vg");
  IG_REQUIRE(!c.fused_fetch || (c.d == 64 || c.d == 128), "fused fetch needs d = 64 or 128");
  if (c.rope_theta > 0.f)
    IG_REQUIRE(buf->Wq && buf->A_cols, "RoPE decoding needs Wq and A_cols");
  else
    IG_REQUIRE(buf->Wq_part, "decoding needs Wq_part");
  IG_REQUIRE(buf->workspace_bytes >= ig_decoder_workspace_bytes(cfg), "decoder workspace too small");
  ig_decoder* d = new ig_decoder();
  d->cfg = c;
  d->buf = *buf;
  d->pool = pool;
  ws_regions(&c, &d->ws_main, &d->ws_sel, &d->ws_fetch);
  const int L = c.layers;
  for (int l = 0; l < L; ++l) {
    const int kl = buf->ks ? buf->ks[l] : c.k;
    if (kl < 1 || kl > c.k) {
      delete d;
      return fail(IG_ERR_INVALID, "layer %d width %d outside [1, config k = %d]", l, kl, c.k);
    }
    d->ks.push_back(kl);
    d->Kpart.push_back(buf->Kpart[l]);
    d->cols.push_back(buf->cols[l]);
    d->Wq_part.push_back(buf->Wq_part ? buf->Wq_part[l] : nullptr);
    d->Wq.push_back(buf->Wq ? buf->Wq[l] : nullptr);
    d->A_cols.push_back(buf->A_cols ? buf->A_cols[l] : nullptr);
  }
  d->buf.Wq_part = nullptr;  // the host arrays belong to the caller; we keep our copies
  d->buf.Wq = nullptr;
  d->buf.A_cols = nullptr;
  d->buf.Kpart = nullptr;
  d->buf.cols = nullptr;
  d->buf.ks = nullptr;
  d->ev_sel.assign(L, nullptr);
  d->ev_got.assign(L, nullptr);
  d->ev_att.assign(L, nullptr);
  cudaError_t e = cudaSuccess;
  for (int l = 0; l < L && e == cudaSuccess; ++l) {
    e = cudaEventCreateWithFlags(&d->ev_sel[l], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d->ev_got[l], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d->ev_att[l], cudaEventDisableTiming);
  }
  if (c.stage_timing) {
    for (auto* v : {&d->tg0, &d->tg1, &d->ts0, &d->ts1, &d->ta0, &d->ta1}) {
      v->assign(2 * L, nullptr);
      for (int l = 0; l < 2 * L && e == cudaSuccess; ++l) e = cudaEventCreate(&(*v)[l]);
    }
  }
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d->ev_fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d->ev_join, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    destroy_events(d);
    delete d;
    return cuda_fail(e, "decoder events");
  }
  if (!error_word()) {  // resolve the error word now, outside any stream capture
    destroy_events(d);
    delete d;
    return fail(IG_ERR_CUDA, "no device error word");
  }
  *out = d;
  return IG_OK;
}

extern "C" ig_status ig_decoder_destroy(ig_decoder* d) {
  if (!d) return IG_OK;
  destroy_events(d);
  delete d;
  return IG_OK;
}

extern "C" ig_status ig_decode_step(ig_decoder* dec, const ig_step_io* io, void* stream,
                                    void* side_stream) {
  IG_REQUIRE(dec && io, "null argument");
  IG_REQUIRE(io->x && io->q && io->k_new && io->v_new && io->L_valid && io->out, "missing step input");
  const ig_decoder_config& c = dec->cfg;
  const ig_decoder_buffers& b = dec->buf;
  IG_REQUIRE(!(c.rope_theta > 0.f) || io->positions, "RoPE decoding needs positions");
  cudaStream_t S = as_stream(stream), G = as_stream(side_stream);
  IG_REQUIRE(S != G, "the fetch stream must differ from the compute stream");
  const int L = c.layers, B = c.B, H = c.H, d = c.d, D = c.D, Lc = c.Lcap;
  const std::vector<int>& ks = dec->ks;
  const size_t xs = (size_t)B * D, ts = (size_t)B * H * d;
  char* ws = static_cast<char*>(b.workspace);
  const size_t spec_att_ws = dec->ws_main;
  void* sel_ws = ws + dec->ws_main;
  const size_t sel_ws_bytes = dec->ws_sel;
  char* fetch_ws = ws + dec->ws_main + dec->ws_sel;
  ig_status st;
  cudaError_t e;

  // G joins S's work so far (the caller's uploads), so it never runs ahead of its inputs
  e = cudaEventRecord(dec->ev_fork, S);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(G, dec->ev_fork, 0);
  if (e != cudaSuccess) return cuda_fail(e, "decode step fork");

  auto attend_append = [&](int l) -> ig_status {
    const size_t buf = (size_t)(l & 1);
    const int32_t* slot = io->slot ? io->slot + (size_t)l * B : nullptr;
    ig_status r;
    if (l == 0) {
      r = ig_dense_attend(S, B, H, d, Lc, c.score_scale, io->q, b.K0, b.V0, io->L_valid, io->k_new,
                          io->v_new, io->out, ws, spec_att_ws);
    } else {
      r = ig_sparse_attend(S, B, H, d, Lc, c.score_scale, io->q + (size_t)l * ts,
                           b.Kg + buf * sz_kv(c), b.Vg + buf * sz_kv(c), b.cnt + (size_t)l * B * H,
                           io->k_new + (size_t)l * ts, io->v_new + (size_t)l * ts,
                           io->out + (size_t)l * ts, ws, spec_att_ws);
    }
    if (r != IG_OK || !slot || c.batched_append || (l > 0 && c.append_on_fetch)) return r;
    if (l == 0)
      return ig_append_kv(S, nullptr, 0, B, H, d, ks[0], Lc, slot, dec->cols[0], io->k_new, io->v_new,
                          dec->Kpart[0], b.K0, b.V0);
    return ig_append_kv(S, dec->pool, l, B, H, d, ks[l], Lc, slot, dec->cols[l],
                        io->k_new + (size_t)l * ts, io->v_new + (size_t)l * ts, dec->Kpart[l],
                        nullptr, nullptr);
  };

  const bool timing = c.stage_timing != 0;
  const int tset = (int)(dec->steps & 1) * L;
  // inside a stream capture the timing events are recorded as external events, which become
  // event-record nodes of the graph (a plain record there would only express a dependency and
  // never fire on replay); outside a capture they are plain records
  cudaStreamCaptureStatus cap_status = cudaStreamCaptureStatusNone;
  if (timing) {
    e = cudaStreamIsCapturing(S, &cap_status);
    if (e != cudaSuccess) return cuda_fail(e, "capture status");
  }
  const unsigned rec_flags = cap_status == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0u;
  auto rec = [&](std::vector<cudaEvent_t>& v, int l, cudaStream_t s) -> cudaError_t {
    return timing ? cudaEventRecordWithFlags(v[tset + l], s, rec_flags) : cudaSuccess;
  };
  auto timed_attend = [&](int l) -> ig_status {
    cudaError_t te = rec(dec->ta0, l, S);
    if (te != cudaSuccess) return cuda_fail(te, "timing event");
    ig_status r = attend_append(l);
    if (r != IG_OK) return r;
    te = rec(dec->ta1, l, S);
    return te == cudaSuccess ? IG_OK : cuda_fail(te, "timing event");
  };
  dec->steps += 1;

  // speculation + selection of layer l on S; G then waits for it
  auto spec_select = [&](int l) -> ig_status {
    float* sc = b.scores;
    int32_t* idx = b.idx + idx_off(c, l);
    int32_t* cnt = b.cnt + (size_t)l * B * H;
    uint8_t* used = b.used ? b.used + (size_t)l * B * Lc : nullptr;
    cudaError_t se = rec(dec->ts0, l, S);
    if (se != cudaSuccess) return cuda_fail(se, "timing event");
    const bool fused = c.fused_select && c.policy == IG_SEL_THRESHOLD && c.cap_frac >= 1.f && Lc <= 8192;
    ig_status r;
    if (fused) {
      const bool rope = c.rope_theta > 0.f;
      r = ig_speculate_select(S, B, D, H, d, ks[l], Lc, io->x + (size_t)(l - 1) * xs,
                              rope ? dec->Wq[l] : dec->Wq_part[l], rope ? dec->A_cols[l] : nullptr,
                              rope ? io->positions : nullptr, c.rope_theta, dec->Kpart[l], io->L_valid,
                              c.score_scale, c.alpha, idx, cnt, used, nullptr, nullptr, ws, spec_att_ws);
    } else if (c.rope_theta > 0.f) {
      r = ig_speculate_rope(S, B, D, H, d, ks[l], Lc, io->x + (size_t)(l - 1) * xs, dec->Wq[l],
                            dec->A_cols[l], io->positions, c.rope_theta, dec->Kpart[l], io->L_valid,
                            c.score_scale, sc, nullptr, ws, spec_att_ws);
    } else {
      r = ig_speculate(S, B, D, H, ks[l], Lc, io->x + (size_t)(l - 1) * xs, dec->Wq_part[l],
                       dec->Kpart[l], io->L_valid, c.score_scale, sc, nullptr, ws, spec_att_ws);
    }
    if (r != IG_OK) return r;
    if (!fused) {
      r = ig_select(S, B, H, Lc, sc, io->L_valid, c.alpha, c.policy, c.cap_frac, idx, cnt, used,
                    sel_ws, sel_ws_bytes);
      if (r != IG_OK) return r;
    }
    se = rec(dec->ts1, l, S);
    if (se == cudaSuccess) se = cudaEventRecord(dec->ev_sel[l], S);
    if (se == cudaSuccess) se = cudaStreamWaitEvent(G, dec->ev_sel[l], 0);
    return se == cudaSuccess ? IG_OK : cuda_fail(se, "decode step events (select)");
  };

  // with batched appends, every layer's token is written in one launch once the step's fetches
  // are done (the fetch stream has joined): the pool rows it may overwrite have been read, and
  // the link carries no fetch while the appends cross it
  auto batched_tail = [&]() -> ig_status {
    if (!c.batched_append || !io->slot) return IG_OK;
    return ig_append_kv_layers(S, dec->pool, L, B, H, d, ks.data(), Lc, io->slot, dec->cols.data(), io->k_new,
                               io->v_new, dec->Kpart.data(), b.K0, b.V0);
  };

  if (L == 1) {
    st = timed_attend(0);
    return st != IG_OK ? st : batched_tail();
  }
  if (c.fused_fetch) {
    // combine(l) and append(l) on S once the fetch stream's partials of layer l are done: the
    // append only then, because the new token may overwrite an evicted slot that the fetch read
    // (speculation(l) has read the partial cache before)
    const size_t fetch_half = dec->ws_fetch / 2;
    std::vector<int> fa_grid(L, 0);
    auto combine_append = [&](int l) -> ig_status {
      cudaError_t ae = cudaStreamWaitEvent(S, dec->ev_att[l], 0);
      if (ae == cudaSuccess) ae = rec(dec->ta0, l, S);
      if (ae != cudaSuccess) return cuda_fail(ae, "decode step wait");
      const size_t off = (size_t)l * ts;
      ig_status r = fetch_attend_combine(S, B, H, d, c.score_scale, io->q + off, io->k_new + off, io->v_new + off,
                                         io->out + off, fetch_ws + (size_t)(l & 1) * fetch_half, fa_grid[l]);
      if (r != IG_OK) return r;
      if (io->slot && !c.batched_append) {
        r = ig_append_kv(S, dec->pool, l, B, H, d, ks[l], Lc, io->slot + (size_t)l * B, dec->cols[l],
                         io->k_new + off, io->v_new + off, dec->Kpart[l], nullptr, nullptr);
        if (r != IG_OK) return r;
      }
      ae = rec(dec->ta1, l, S);
      return ae == cudaSuccess ? IG_OK : cuda_fail(ae, "timing event");
    };
    for (int l = 1; l < L; ++l) {
      if (l >= 3) {  // attention(l-2) yields layer l-1's input, which speculation(l) reads
        st = combine_append(l - 2);
        if (st != IG_OK) return st;
      }
      st = spec_select(l);
      if (st != IG_OK) return st;
      // the partial set l % 2 was last read by combine(l-2), which S ran before selection(l)
      e = rec(dec->tg0, l, G);
      if (e != cudaSuccess) return cuda_fail(e, "timing event");
      const size_t off = (size_t)l * ts;
      st = fetch_attend_partials(G, dec->pool, l, B, H, d, Lc, c.score_scale, io->q + off, b.idx + idx_off(c, l),
                                 b.cnt + (size_t)l * B * H, io->k_new + off, io->v_new + off, io->out + off,
                                 fetch_ws + (size_t)(l & 1) * fetch_half, fetch_half, c.gather_ctas, &fa_grid[l]);
      if (st != IG_OK) return st;
      e = rec(dec->tg1, l, G);
      if (e == cudaSuccess) e = cudaEventRecord(dec->ev_att[l], G);
      if (e != cudaSuccess) return cuda_fail(e, "decode step events (fetch)");
      if (l == 1) {
        st = timed_attend(0);
        if (st != IG_OK) return st;
      }
    }
    for (int l = L - 2 > 1 ? L - 2 : 1; l < L; ++l) {
      st = combine_append(l);
      if (st != IG_OK) return st;
    }
    e = cudaEventRecord(dec->ev_join, G);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(S, dec->ev_join, 0);
    if (e != cudaSuccess) return cuda_fail(e, "decode step join");
    return batched_tail();
  }
  for (int l = 1; l < L; ++l) {
    st = spec_select(l);
    if (st != IG_OK) return st;
    const int32_t* idx = b.idx + idx_off(c, l);
    const int32_t* cnt = b.cnt + (size_t)l * B * H;
    if (l >= 3) e = cudaStreamWaitEvent(G, dec->ev_att[l - 2], 0);
    if (e == cudaSuccess) e = rec(dec->tg0, l, G);
    if (e != cudaSuccess) return cuda_fail(e, "decode step events (select)");
    const size_t buf = (size_t)(l & 1);
    st = ig_gather_kv(G, dec->pool, l, B, H, d, Lc, idx, cnt, b.Kg + buf * sz_kv(c),
                      b.Vg + buf * sz_kv(c), c.gather_ctas);
    if (st != IG_OK) return st;
    e = rec(dec->tg1, l, G);
    if (e == cudaSuccess) e = cudaEventRecord(dec->ev_got[l], G);
    if (e != cudaSuccess) return cuda_fail(e, "decode step events (gather)");
    if (c.append_on_fetch && !c.batched_append && io->slot) {
      // the fetch stream writes layer l's new token right after reading layer l's rows: no fetch
      // of its own is in flight then, and the compute stream is spared the host stores
      st = ig_append_kv(G, dec->pool, l, B, H, d, ks[l], Lc, io->slot + (size_t)l * B, dec->cols[l],
                        io->k_new + (size_t)l * ts, io->v_new + (size_t)l * ts, dec->Kpart[l], nullptr, nullptr);
      if (st != IG_OK) return st;
    }
    // layer l-1 attends while layer l is fetched (layer 0 needs no fetch)
    if (l >= 2) {
      e = cudaStreamWaitEvent(S, dec->ev_got[l - 1], 0);
      if (e != cudaSuccess) return cuda_fail(e, "decode step wait");
    }
    st = timed_attend(l - 1);
    if (st != IG_OK) return st;
    e = cudaEventRecord(dec->ev_att[l - 1], S);
    if (e != cudaSuccess) return cuda_fail(e, "decode step events (attend)");
  }
  if (L >= 2) {
    e = cudaStreamWaitEvent(S, dec->ev_got[L - 1], 0);
    if (e != cudaSuccess) return cuda_fail(e, "decode step wait");
    st = timed_attend(L - 1);
    if (st != IG_OK) return st;
  }
  // S ends after everything G did, so the caller can treat S alone as the step's stream
  e = cudaEventRecord(dec->ev_join, G);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(S, dec->ev_join, 0);
  if (e != cudaSuccess) return cuda_fail(e, "decode step join");
  return batched_tail();
}

extern "C" ig_status ig_decoder_stage_ms(ig_decoder* dec, int steps_back, float* ms_out,
                                         int* counts_out) {
  IG_REQUIRE(dec && ms_out, "null argument");
  IG_REQUIRE(steps_back == 0 || steps_back == 1, "steps_back must be 0 or 1");
  IG_REQUIRE(dec->cfg.stage_timing && dec->steps > steps_back, "stage timing is off or no such step");
  const int L = dec->cfg.layers;
  const int tset = (int)((dec->steps - 1 - steps_back) & 1) * L;
  double sums[4] = {0, 0, 0, 0};
  int counts[4] = {0, 0, 0, 0};
  auto span = [&](cudaEvent_t a, cudaEvent_t b, int which) -> cudaError_t {
    cudaError_t e = cudaEventSynchronize(b);
    if (e != cudaSuccess) return e;
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, a, b);
    if (e != cudaSuccess) return e;
    sums[which] += ms;
    counts[which] += 1;
    return cudaSuccess;
  };
  cudaError_t e = cudaSuccess;
  for (int l = 0; l < L && e == cudaSuccess; ++l) {
    if (l >= 1) e = span(dec->tg0[tset + l], dec->tg1[tset + l], 0);
    if (e == cudaSuccess && l >= 1) e = span(dec->ts0[tset + l], dec->ts1[tset + l], 1);
    if (e == cudaSuccess) e = span(dec->ta0[tset + l], dec->ta1[tset + l], l == 0 ? 3 : 2);
  }
  if (e != cudaSuccess) return cuda_fail(e, "stage timing");
  for (int i = 0; i < 4; ++i) {
    ms_out[i] = (float)sums[i];
    if (counts_out) counts_out[i] = counts[i];
  }
  return IG_OK;
}

extern "C" ig_status ig_decoder_timeline(ig_decoder* dec, int steps_back, float* t_out) {
  IG_REQUIRE(dec && t_out, "null argument");
  IG_REQUIRE(steps_back == 0 || steps_back == 1, "steps_back must be 0 or 1");
  IG_REQUIRE(dec->cfg.stage_timing && dec->steps > steps_back, "stage timing is off or no such step");
  const int L = dec->cfg.layers;
  const int tset = (int)((dec->steps - 1 - steps_back) & 1) * L;
  // the step's first timed stage: speculation of layer 1 (layer 0's attention when L == 1)
  cudaEvent_t t0 = L > 1 ? dec->ts0[tset + 1] : dec->ta0[tset];
  const float nan = std::numeric_limits<float>::quiet_NaN();
  cudaError_t e = cudaSuccess;
  auto at = [&](cudaEvent_t ev, float* out) -> cudaError_t {
    cudaError_t r = cudaEventSynchronize(ev);
    if (r == cudaSuccess) r = cudaEventElapsedTime(out, t0, ev);
    return r;
  };
  for (int l = 0; l < L && e == cudaSuccess; ++l) {
    float* row = t_out + (size_t)l * 6;
    for (int j = 0; j < 4; ++j) row[j] = nan;
    if (l >= 1) {
      e = at(dec->tg0[tset + l], &row[0]);
      if (e == cudaSuccess) e = at(dec->tg1[tset + l], &row[1]);
      if (e == cudaSuccess) e = at(dec->ts0[tset + l], &row[2]);
      if (e == cudaSuccess) e = at(dec->ts1[tset + l], &row[3]);
    }
    if (e == cudaSuccess) e = at(dec->ta0[tset + l], &row[4]);
    if (e == cudaSuccess) e = at(dec->ta1[tset + l], &row[5]);
  }
  return e == cudaSuccess ? IG_OK : cuda_fail(e, "stage timeline");
}

extern "C" ig_status ig_decoder_graph_capture(ig_decoder* dec, const ig_step_io* io, void* stream,
                                              void* side_stream) {
  IG_REQUIRE(dec && io, "null argument");
  cudaStream_t S = as_stream(stream);
  IG_REQUIRE(S != nullptr, "graph capture needs a created (non-default) compute stream");
  for (cudaGraphExec_t& g : dec->graph)
    if (g) {
      cudaGraphExecDestroy(g);
      g = nullptr;
    }
  const long long saved = dec->steps;
  const int n = dec->cfg.stage_timing ? 2 : 1;
  for (int p = 0; p < n; ++p) {
    dec->steps = p;  // selects timing-event set p
    const uint64_t k0 = ig_launch_count();
    cudaError_t e = cudaStreamBeginCapture(S, cudaStreamCaptureModeRelaxed);
    if (e != cudaSuccess) {
      dec->steps = saved;
      return cuda_fail(e, "begin capture");
    }
    const ig_status st = ig_decode_step(dec, io, stream, side_stream);
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(S, &graph);
    const uint64_t captured = ig_launch_count() - k0;
    count_launches(-(int64_t)captured);  // captured launches have not run
    if (st != IG_OK || e != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      dec->steps = saved;
      return st != IG_OK ? st : cuda_fail(e, "end capture");
    }
    e = cudaGraphInstantiate(&dec->graph[p], graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
      dec->steps = saved;
      return cuda_fail(e, "graph instantiate");
    }
    dec->graph_kernels = captured;
  }
  dec->steps = saved;
  return IG_OK;
}

extern "C" ig_status ig_decoder_graph_launch(ig_decoder* dec, void* stream) {
  IG_REQUIRE(dec, "null decoder");
  const int p = dec->cfg.stage_timing ? (int)(dec->steps & 1) : 0;
  IG_REQUIRE(dec->graph[p], "no captured step (call ig_decoder_graph_capture first)");
  cudaError_t e = cudaGraphLaunch(dec->graph[p], as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "graph launch");
  dec->steps += 1;
  count_launches((int64_t)dec->graph_kernels);
  return IG_OK;
}
