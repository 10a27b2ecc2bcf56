// Part of layer.cu's translation unit (included inside its anonymous
// namespace, after the plan, the launcher and the layer's stage loops): the
// layer on sequence chunks inside the head stages.

// ---------------------------------------------------------------------------
// Head stages combined with sequence chunks ("Untied Ulysses" summary page,
// Limitations and Future directions: FPDT chunks the sequence, UPipe the
// heads, and the two compose).  The sequence is cut into n_c chunks of
// Sc = S / n_c tokens; per chunk i (forward: ascending) and stage s the
// chunk's rows are projected onto the stage's heads and exchanged; the
// chunk's K and V go to an offload store (device or page-locked host memory,
// the caller's) and the queries attend to KV chunks 0..i, each fetched from
// the store into one of two device windows on a copy stream while the tensor
// cores work on the previous one; the partial results merge by log-sum-exp
// in the attention epilogue.  Every device buffer is O(Sc), not O(S).
// Backward: the K/V chunks are recomputed into the store, then query chunks
// run in descending order, so a KV chunk's gradient is complete when its own
// query chunk is done; partial dK/dV of the chunks in between live in the
// store next to K and V.
// ---------------------------------------------------------------------------
struct ChunkPlan {
  Plan base;                 // the in-order head stages
  int n_c = 0, Sc = 0, nkv = 0;
  std::vector<int> kv_first_stage, kv_last_stage;  // per KV head
  size_t off_seq = 0, off_qkvh = 0, off_kvw[2] = {0, 0}, off_dkvw[2] = {0, 0};
  size_t off_oacc = 0, off_lacc = 0, off_doh = 0, off_dsum = 0, off_lse2 = 0, off_dq = 0, off_acc32 = 0;
  size_t arena = 0, persistent = 0, total = 0, store = 0;
};

// CTAs per KV block of a chunk-pair attention backward: the split (1..8)
// whose grid fills its last wave of SMs best (ties to the smaller split)
int choose_q_split(long long ctas) {
  const double sms = num_sms();
  int best = 1;
  double best_eff = 0.0;
  for (int q = 1; q <= 8; ++q) {
    const double waves = static_cast<double>(ctas) * q / sms;
    const double eff = waves / std::ceil(waves);
    if (eff > best_eff + 0.02) {
      best = q;
      best_eff = eff;
    }
  }
  return best;
}

int check_chunks(const Shape& s, int n_c) {
  int rc = check_shape(s);
  if (rc != UPIPE_OK) return rc;
  if (s.sched != UPIPE_SCHED_INORDER || n_c <= 0 || s.S % n_c) return UPIPE_EINVAL;
  const int Sc = s.S / n_c;
  if (Sc % 128 || Sc % s.C) return UPIPE_EINVAL;
  return UPIPE_OK;
}

ChunkPlan make_chunk_plan(const Shape& s, int n_c, bool backward) {
  ChunkPlan c;
  c.base.sh = s;
  build_schedule(c.base);
  c.n_c = n_c;
  c.Sc = s.S / n_c;
  c.kv_first_stage.assign(s.G, -1);
  c.kv_last_stage.assign(s.G, -1);
  for (int i = 0; i < c.base.n_stages; ++i)
    for (int g : c.base.st[i].kv_proj) {
      if (c.kv_first_stage[g] < 0) c.kv_first_stage[g] = i;
      c.kv_last_stage[g] = i;
      c.nkv = std::max<int>(c.nkv, static_cast<int>(c.base.st[i].kv_proj.size()));
    }
  const size_t Sc = c.Sc, d = s.d, U = s.U, nkv = c.nkv;
  const int max_cols = static_cast<int>(U + 2 * nkv);
  size_t o = 0;
  c.off_seq = o;
  o = align256(o + Sc * max_cols * d * 2);
  c.off_qkvh = o;
  o = align256(o + (backward ? U : U + 2 * nkv) * Sc * d * 2);
  for (int b = 0; b < 2; ++b) {
    c.off_kvw[b] = o;
    o = align256(o + 2 * nkv * Sc * d * 2);
  }
  if (backward) {
    for (int b = 0; b < 2; ++b) {
      c.off_dkvw[b] = o;
      o = align256(o + 2 * nkv * Sc * d * 4);
    }
    c.off_doh = o;
    o = align256(o + U * Sc * d * 2);
    c.off_dsum = o;
    o = align256(o + U * Sc * 4);
    c.off_lse2 = o;
    o = align256(o + U * Sc * 4);
    c.off_dq = o;
    o = align256(o + U * Sc * d * 4);
  } else {
    c.off_oacc = o;
    o = align256(o + U * Sc * d * 4);
    c.off_lacc = o;
    o = align256(o + U * Sc * 4);
  }
  c.arena = o;
  c.off_acc32 = o;
  if (c.base.n_stages > 1) o = align256(o + Sc * s.dm * 4);
  c.persistent = o - c.arena;
  c.total = o;
  // store: [chunk][K, V][G][Sc][d] bf16, then (backward) the same in fp32 for dK, dV
  c.store = static_cast<size_t>(s.S) * 2 * s.G * d * (backward ? 2 + 4 : 2);
  return c;
}

// The copy stream and the events of one chunked call.
struct ChunkStreams {
  cudaStream_t main = nullptr, cs = nullptr;
  cudaEvent_t ev[8] = {};
  size_t copied = 0;
  cudaError_t err = cudaSuccess;
  cudaEvent_t* ready() { return ev; }          // [2] window filled (copy stream)
  cudaEvent_t* mainfree() { return ev + 2; }   // [2] window's last device use issued (main)
  cudaEvent_t* produced() { return ev + 4; }   // [2] a chunk to store is in its buffer (main)
  cudaEvent_t* stored() { return ev + 6; }     // [2] that buffer has been copied out (copy stream)
  bool init(cudaStream_t m) {
    main = m;
    cs = side_stream();
    if (!cs) return false;
    for (cudaEvent_t& e : ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
    // nothing the copy stream does may start before the caller's prior work
    if (cudaEventRecord(ev[4], main) != cudaSuccess || cudaStreamWaitEvent(cs, ev[4], 0) != cudaSuccess) return false;
    return true;
  }
  void copy(void* dst, const void* src, size_t bytes) {
    if (err != cudaSuccess) return;
    err = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, cs);
    copied += bytes;
  }
  void record(cudaEvent_t e, cudaStream_t s) {
    if (err == cudaSuccess) err = cudaEventRecord(e, s);
  }
  void wait(cudaStream_t s, cudaEvent_t e) {
    if (err == cudaSuccess) err = cudaStreamWaitEvent(s, e, 0);
  }
  void finish() {
    // the caller's stream ends after every copy
    if (cs && ev[0]) {
      record(ev[0], cs);
      wait(main, ev[0]);
    }
    for (cudaEvent_t e : ev)
      if (e) cudaEventDestroy(e);
  }
};

int chunk_finish(Launcher& L, ChunkStreams& cst, const ChunkPlan& c, upipe_stats* stats) {
  cst.finish();
  if (stats) {
    Plan p = c.base;
    p.arena = c.arena;
    p.persistent = c.persistent;
    finish(L, p, stats);
    stats->offload_bytes = c.store;
    stats->offload_copy_bytes = cst.copied;
  }
  if (cst.err != cudaSuccess) return UPIPE_ECUDA;
  return L.ok() ? UPIPE_OK : UPIPE_ECUDA;
}

int chunk_checks(const Shape& s, int n_c, const void* const* ptrs, int n_ptrs, const void* ws, size_t ws_bytes,
                 const ChunkPlan& c, const void* store, size_t store_bytes) {
  int rc = check_chunks(s, n_c);
  if (rc != UPIPE_OK) return rc;
  rc = common_checks(s, ptrs, n_ptrs, ws, ws_bytes, c.total);
  if (rc != UPIPE_OK) return rc;
  if (!store || !aligned16(store)) return UPIPE_EINVAL;
  if (store_bytes < c.store) return UPIPE_ENOSPC;
  return UPIPE_OK;
}

int attn_fwd_chunked_issue(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model,
                           int H, int G, int d_head, int U, int C, int n_c, upipe_bf16* Y, upipe_bf16* O_saved,
                           float* lse, void* ws, size_t ws_bytes, void* store, size_t store_bytes, void* stream,
                           upipe_stats* stats) {
  const Shape s{S, d_model, H, G, d_head, U, C, UPIPE_SCHED_INORDER};
  int rc = check_chunks(s, n_c);
  if (rc != UPIPE_OK) return rc;
  const ChunkPlan c = make_chunk_plan(s, n_c, false);
  const void* ptrs[] = {X, W_qkv, W_o, Y, O_saved, lse};
  rc = chunk_checks(s, n_c, ptrs, 6, ws, ws_bytes, c, store, store_bytes);
  if (rc != UPIPE_OK) return rc;
  ChunkStreams cst;
  Launcher L{static_cast<cudaStream_t>(stream), status_ptr()};
  if (!cst.init(L.st)) {
    cst.finish();
    return UPIPE_ECUDA;
  }
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int d = d_head, Sc = c.Sc, n_st = c.base.n_stages;
  const size_t chunk_elems = static_cast<size_t>(Sc) * d;  // one head of one chunk
  uint16_t* seq = reinterpret_cast<uint16_t*>(w + c.off_seq);
  uint16_t* qkvh = reinterpret_cast<uint16_t*>(w + c.off_qkvh);
  float* oacc = reinterpret_cast<float*>(w + c.off_oacc);
  float* lacc = reinterpret_cast<float*>(w + c.off_lacc);
  float* y32 = reinterpret_cast<float*>(w + c.off_acc32);
  uint16_t* kst = static_cast<uint16_t*>(store);
  auto store_at = [&](int j, int part, int g) { return kst + ((static_cast<size_t>(j) * 2 + part) * G + g) * chunk_elems; };
  int n_fetch = 0;  // fetches so far: window n_fetch & 1
  for (int i = 0; i < n_c && L.ok() && cst.err == cudaSuccess; ++i) {
    const size_t row0 = static_cast<size_t>(i) * Sc;
    for (int si = 0; si < n_st && L.ok(); ++si) {
      const Stage& g = c.base.st[si];
      const int nkv = static_cast<int>(g.kv_proj.size());
      const int g0 = g.kv_proj[0];
      // fetch of KV chunk j of this stage into the next window
      auto fetch = [&](int j) {
        const int b = n_fetch & 1;
        uint16_t* kw = reinterpret_cast<uint16_t*>(w + c.off_kvw[b]);
        cst.wait(cst.cs, cst.mainfree()[b]);
        cst.copy(kw, store_at(j, 0, g0), nkv * chunk_elems * 2);
        cst.copy(kw + nkv * chunk_elems, store_at(j, 1, g0), nkv * chunk_elems * 2);
        cst.record(cst.ready()[b], cst.cs);
        ++n_fetch;
      };
      const int fetch_base = n_fetch;
      if (i > 0) fetch(0);
      // (1) projection of the chunk's rows, (2) exchange: Q slots, then K and V
      // (one slot per KV head), into qkvh once its K/V have left for the store
      GemmDesc gd;
      gd.A = X + row0 * d_model; gd.lda = d_model; gd.a_rows = Sc; gd.a_cols = d_model; gd.a_mn = false;
      gd.B = W_qkv; gd.ldb = static_cast<long long>(H + 2 * G) * d; gd.b_rows = d_model; gd.b_cols = gd.ldb;
      gd.b_mn = true;
      gd.M = Sc; gd.N = (U + 2 * nkv) * d; gd.K = d_model;
      head_blocks(gd.bmap_n, stage_wqkv_heads(s, g.q_heads, g.kv_proj), d);
      gd.out = seq; gd.ldo = static_cast<long long>(U + 2 * nkv) * d; gd.out_mode = kOutBf16;
      L.gemm(gd);
      cst.wait(L.st, cst.stored()[0]);
      Seq2HeadDesc x;
      x.src = seq; x.ld_src = gd.ldo; x.dst = qkvh; x.S = Sc; x.D = d;
      x.n_slots = U + 2 * nkv;
      for (int k = 0; k < x.n_slots; ++k) x.src_head[k] = static_cast<uint16_t>(k);
      L.s2h(x);
      // the chunk's K and V to the store
      cst.record(cst.produced()[0], L.st);
      cst.wait(cst.cs, cst.produced()[0]);
      cst.copy(store_at(i, 0, g0), qkvh + static_cast<size_t>(U) * chunk_elems, nkv * chunk_elems * 2);
      cst.copy(store_at(i, 1, g0), qkvh + static_cast<size_t>(U + nkv) * chunk_elems, nkv * chunk_elems * 2);
      cst.record(cst.stored()[0], cst.cs);
      // (3) attention: the diagonal chunk from qkvh, then chunks 0..i-1 from the windows
      AttnFwdDesc a;
      a.Q = qkvh;
      a.O = seq;  // the sequence buffer is dead after the exchange
      a.lse = lse + row0; a.lse_ld = S;
      a.S = Sc; a.D = d; a.n_qslots = U; a.n_kvslots = nkv;
      a.kv_len = Sc; a.kv_ld = Sc;
      a.o_acc = oacc; a.lse_acc = lacc;
      for (int k = 0; k < U; ++k) {
        a.kv_slot[k] = static_cast<uint16_t>(std::find(g.kv_proj.begin(), g.kv_proj.end(), kv_of(s, g.q_heads[k])) -
                                             g.kv_proj.begin());
        a.lse_row[k] = static_cast<uint16_t>(g.q_heads[k]);
      }
      a.K = qkvh + static_cast<size_t>(U) * chunk_elems;
      a.V = qkvh + static_cast<size_t>(U + nkv) * chunk_elems;
      a.q_off = 0;
      a.mode = i == 0 ? kFwdPlain : kFwdFirst;
      L.fwd(a);
      for (int j = 0; j < i && L.ok(); ++j) {
        const int n = fetch_base + j, b = n & 1;
        if (j + 1 < i) fetch(j + 1);
        uint16_t* kw = reinterpret_cast<uint16_t*>(w + c.off_kvw[b]);
        cst.wait(L.st, cst.ready()[b]);
        a.K = kw;
        a.V = kw + static_cast<size_t>(nkv) * chunk_elems;
        a.q_off = (i - j) * Sc;
        a.mode = j + 1 == i ? kFwdLast : kFwdMiddle;
        L.fwd(a);
        cst.record(cst.mainfree()[b], L.st);
      }
      // (4) exchange back into the chunk's rows of O_saved
      Head2SeqDesc hb;
      hb.src = seq; hb.src_f32 = false;
      hb.dst = O_saved + row0 * H * d; hb.ld_dst = static_cast<long long>(H) * d;
      hb.S = Sc; hb.D = d; hb.n_heads = U;
      for (int k = 0; k <= U; ++k) hb.first[k] = static_cast<uint16_t>(k);
      for (int k = 0; k < U; ++k) {
        hb.dst_head[k] = static_cast<uint16_t>(g.q_heads[k]);
        hb.src_slot[k] = static_cast<uint16_t>(k);
      }
      L.h2s(hb);
      // (5) the stage's share of the chunk's rows of Y
      GemmDesc go;
      go.A = O_saved + row0 * H * d; go.lda = static_cast<long long>(H) * d; go.a_rows = Sc; go.a_cols = go.lda;
      go.a_mn = false;
      go.B = W_o; go.ldb = d_model; go.b_rows = static_cast<long long>(H) * d; go.b_cols = d_model; go.b_mn = true;
      go.M = Sc; go.N = d_model; go.K = U * d;
      head_blocks(go.amap_k, g.q_heads, d);
      go.bmap_k = go.amap_k;
      upipe_bf16* Yc = Y + row0 * d_model;
      if (n_st == 1) {
        go.out = Yc; go.ldo = d_model; go.out_mode = kOutBf16;
      } else if (si == 0) {
        go.out = y32; go.ldo = d_model; go.out_mode = kOutF32;
      } else if (si + 1 < n_st) {
        go.out = y32; go.ldo = d_model; go.out_mode = kOutF32Acc;
      } else {
        go.out = Yc; go.ldo = d_model; go.out_mode = kOutBf16PlusF32; go.aux = y32; go.ld_aux = d_model;
      }
      L.gemm(go);
    }
  }
  return chunk_finish(L, cst, c, stats);
}

int attn_bwd_chunked_issue(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model,
                           int H, int G, int d_head, int U, int C, int n_c, const upipe_bf16* O_saved,
                           const float* lse, const upipe_bf16* dY, upipe_bf16* dX, float* dW_qkv, float* dW_o,
                           void* ws, size_t ws_bytes, void* store, size_t store_bytes, void* stream,
                           upipe_stats* stats) {
  const Shape s{S, d_model, H, G, d_head, U, C, UPIPE_SCHED_INORDER};
  int rc = check_chunks(s, n_c);
  if (rc != UPIPE_OK) return rc;
  const ChunkPlan c = make_chunk_plan(s, n_c, true);
  const void* ptrs[] = {X, W_qkv, W_o, O_saved, lse, dY, dX, dW_qkv, dW_o};
  rc = chunk_checks(s, n_c, ptrs, 9, ws, ws_bytes, c, store, store_bytes);
  if (rc != UPIPE_OK) return rc;
  ChunkStreams cst;
  Launcher L{static_cast<cudaStream_t>(stream), status_ptr()};
  if (!cst.init(L.st)) {
    cst.finish();
    return UPIPE_ECUDA;
  }
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int d = d_head, Sc = c.Sc, n_st = c.base.n_stages;
  const size_t chunk_elems = static_cast<size_t>(Sc) * d;
  const long long qkv_ld = static_cast<long long>(H + 2 * G) * d;
  uint16_t* seq = reinterpret_cast<uint16_t*>(w + c.off_seq);
  uint16_t* qh = reinterpret_cast<uint16_t*>(w + c.off_qkvh);
  uint16_t* doh = reinterpret_cast<uint16_t*>(w + c.off_doh);
  float* dsum = reinterpret_cast<float*>(w + c.off_dsum);
  float* lse2 = reinterpret_cast<float*>(w + c.off_lse2);
  float* dq = reinterpret_cast<float*>(w + c.off_dq);
  float* dx32 = reinterpret_cast<float*>(w + c.off_acc32);
  uint16_t* kst = static_cast<uint16_t*>(store);
  float* dst = reinterpret_cast<float*>(static_cast<uint8_t*>(store) + static_cast<size_t>(S) * 2 * G * d * 2);
  auto kv_at = [&](int j, int part, int g) { return kst + ((static_cast<size_t>(j) * 2 + part) * G + g) * chunk_elems; };
  auto dkv_at = [&](int j, int part, int g) { return dst + ((static_cast<size_t>(j) * 2 + part) * G + g) * chunk_elems; };

  if (cudaMemsetAsync(dW_qkv, 0, static_cast<size_t>(d_model) * qkv_ld * 4, L.st) != cudaSuccess) {
    cst.finish();
    return UPIPE_ECUDA;
  }
  // (a) every K/V chunk of every stage into the store, through the two windows
  int n_buf = 0;
  for (int j = 0; j < n_c && L.ok(); ++j)
    for (int si = 0; si < n_st && L.ok(); ++si) {
      const Stage& g = c.base.st[si];
      const int nkv = static_cast<int>(g.kv_proj.size());
      if (c.kv_first_stage[g.kv_proj[0]] != si) continue;  // projected by an earlier stage
      const int b = n_buf++ & 1;
      uint16_t* kw = reinterpret_cast<uint16_t*>(w + c.off_kvw[b]);
      std::vector<int> heads;
      for (int part = 0; part < 2; ++part)
        for (int m = 0; m < nkv; ++m) heads.push_back((part == 0 ? H : H + G) + g.kv_proj[m]);
      GemmDesc gd;
      gd.A = X + static_cast<size_t>(j) * Sc * d_model; gd.lda = d_model; gd.a_rows = Sc; gd.a_cols = d_model;
      gd.a_mn = false;
      gd.B = W_qkv; gd.ldb = qkv_ld; gd.b_rows = d_model; gd.b_cols = qkv_ld; gd.b_mn = true;
      gd.M = Sc; gd.N = 2 * nkv * d; gd.K = d_model;
      head_blocks(gd.bmap_n, heads, d);
      gd.out = seq; gd.ldo = static_cast<long long>(2 * nkv) * d; gd.out_mode = kOutBf16;
      L.gemm(gd);
      cst.wait(L.st, cst.stored()[b]);
      Seq2HeadDesc x;
      x.src = seq; x.ld_src = gd.ldo; x.dst = kw; x.S = Sc; x.D = d; x.n_slots = 2 * nkv;
      for (int k = 0; k < x.n_slots; ++k) x.src_head[k] = static_cast<uint16_t>(k);
      L.s2h(x);
      cst.record(cst.produced()[b], L.st);
      cst.wait(cst.cs, cst.produced()[b]);
      cst.copy(kv_at(j, 0, g.kv_proj[0]), kw, nkv * chunk_elems * 2);
      cst.copy(kv_at(j, 1, g.kv_proj[0]), kw + nkv * chunk_elems, nkv * chunk_elems * 2);
      cst.record(cst.stored()[b], cst.cs);
    }
  // the fetches below run on the copy stream after these copies

  // (b) query chunks, last first
  int n_fetch = 0;
  for (int i = n_c - 1; i >= 0 && L.ok() && cst.err == cudaSuccess; --i) {
    const size_t row0 = static_cast<size_t>(i) * Sc;
    int dx_done = 0;
    for (int si = 0; si < n_st && L.ok(); ++si) {
      const Stage& g = c.base.st[si];
      const int nkv = static_cast<int>(g.kv_proj.size());
      const int g0 = g.kv_proj[0];
      // partial dK/dV of this stage's KV heads exist in the store unless this
      // is the first visit of those heads (last query chunk, first stage)
      const bool acc = i < n_c - 1 || c.kv_first_stage[g0] < si;
      const bool final_here = c.kv_last_stage[g0] == si;  // chunk i's dK, dV complete after j = i
      auto fetch = [&](int j) {
        const int b = n_fetch++ & 1;
        uint16_t* kw = reinterpret_cast<uint16_t*>(w + c.off_kvw[b]);
        float* dkw = reinterpret_cast<float*>(w + c.off_dkvw[b]);
        cst.wait(cst.cs, cst.mainfree()[b]);
        cst.copy(kw, kv_at(j, 0, g0), nkv * chunk_elems * 2);
        cst.copy(kw + nkv * chunk_elems, kv_at(j, 1, g0), nkv * chunk_elems * 2);
        if (acc) {
          cst.copy(dkw, dkv_at(j, 0, g0), nkv * chunk_elems * 4);
          cst.copy(dkw + nkv * chunk_elems, dkv_at(j, 1, g0), nkv * chunk_elems * 4);
        }
        cst.record(cst.ready()[b], cst.cs);
      };
      const int fetch_base = n_fetch;
      fetch(i);  // pairs run j = i, i-1, ..., 0
      // Q of the chunk, then dO = dY W_o[rows of the stage]^T, both to head layout
      GemmDesc gq;
      gq.A = X + row0 * d_model; gq.lda = d_model; gq.a_rows = Sc; gq.a_cols = d_model; gq.a_mn = false;
      gq.B = W_qkv; gq.ldb = qkv_ld; gq.b_rows = d_model; gq.b_cols = qkv_ld; gq.b_mn = true;
      gq.M = Sc; gq.N = U * d; gq.K = d_model;
      head_blocks(gq.bmap_n, g.q_heads, d);
      gq.out = seq; gq.ldo = static_cast<long long>(U) * d; gq.out_mode = kOutBf16;
      L.gemm(gq);
      Seq2HeadDesc xq;
      xq.src = seq; xq.ld_src = gq.ldo; xq.dst = qh; xq.S = Sc; xq.D = d; xq.n_slots = U;
      for (int k = 0; k < U; ++k) xq.src_head[k] = static_cast<uint16_t>(k);
      L.s2h(xq);
      GemmDesc gd;
      gd.A = dY + row0 * d_model; gd.lda = d_model; gd.a_rows = Sc; gd.a_cols = d_model; gd.a_mn = false;
      gd.B = W_o; gd.ldb = d_model; gd.b_rows = static_cast<long long>(H) * d; gd.b_cols = d_model; gd.b_mn = false;
      gd.M = Sc; gd.N = U * d; gd.K = d_model;
      head_blocks(gd.bmap_n, g.q_heads, d);
      gd.out = seq; gd.ldo = static_cast<long long>(U) * d; gd.out_mode = kOutBf16;
      L.gemm(gd);
      Seq2HeadDesc xd = xq;
      xd.dst = doh;
      L.s2h(xd);
      BwdPrepDesc pr;
      pr.dO = seq; pr.ld_do = static_cast<long long>(U) * d;
      pr.O = O_saved + row0 * H * d; pr.ld_o = static_cast<long long>(H) * d;
      pr.lse = lse + row0; pr.lse_ld = S;
      pr.Dsum = dsum; pr.lse2 = lse2; pr.dQacc = dq;
      pr.S = Sc; pr.D = d; pr.n_slots = U;
      for (int k = 0; k < U; ++k) {
        pr.do_unit[k] = k;
        pr.o_unit[k] = g.q_heads[k];
        pr.lse_row[k] = static_cast<uint16_t>(g.q_heads[k]);
      }
      L.prep(pr);
      // sequence buffer of the stage's gradients: dQ, then (when complete) dK, dV
      const int n_out = U + (final_here ? 2 * nkv : 0);
      const long long ld_dseq = static_cast<long long>(n_out) * d;
      AttnBwdDesc ab;
      ab.Q = qh; ab.dO = doh; ab.lse2 = lse2; ab.Dsum = dsum; ab.dQacc = dq;
      ab.S = Sc; ab.D = d; ab.n_qslots = U; ab.n_kvslots = nkv;
      ab.kv_len = Sc; ab.kv_ld = Sc;
      ab.accumulate_kv = acc ? 1 : 0;
      ab.q_split = choose_q_split(static_cast<long long>(nkv) * (Sc / 128));
      for (int k = 0; k < U; ++k)
        ab.kv_slot[k] = static_cast<uint16_t>(std::find(g.kv_proj.begin(), g.kv_proj.end(), kv_of(s, g.q_heads[k])) -
                                              g.kv_proj.begin());
      for (int j = i; j >= 0 && L.ok(); --j) {
        const int n = fetch_base + (i - j), b = n & 1;
        if (j > 0) fetch(j - 1);
        uint16_t* kw = reinterpret_cast<uint16_t*>(w + c.off_kvw[b]);
        float* dkw = reinterpret_cast<float*>(w + c.off_dkvw[b]);
        cst.wait(L.st, cst.ready()[b]);
        if (ab.q_split > 1 && !acc && L.ok() &&
            cudaMemsetAsync(dkw, 0, static_cast<size_t>(2 * nkv) * chunk_elems * 4, L.st) != cudaSuccess)
          L.err = cudaErrorUnknown;  // the split CTAs add their dK, dV into zeros
        ab.K = kw;
        ab.V = kw + static_cast<size_t>(nkv) * chunk_elems;
        ab.dK = dkw;
        ab.dV = dkw + static_cast<size_t>(nkv) * chunk_elems;
        ab.q_off = (i - j) * Sc;
        L.bwd(ab);
        const bool done = (j == i) && final_here;
        if (done) {
          // dK, dV of chunk i are complete: fp32 -> bf16 into the sequence buffer
          Head2SeqDesc hb;
          hb.src = dkw; hb.src_f32 = true;
          hb.dst = seq; hb.ld_dst = ld_dseq; hb.S = Sc; hb.D = d; hb.n_heads = 2 * nkv;
          for (int k = 0; k < 2 * nkv; ++k) {
            hb.dst_head[k] = static_cast<uint16_t>(U + k);
            hb.src_slot[k] = static_cast<uint16_t>(k);
            hb.first[k] = static_cast<uint16_t>(k);
          }
          hb.first[2 * nkv] = static_cast<uint16_t>(2 * nkv);
          L.h2s(hb);
        }
        cst.record(cst.mainfree()[b], L.st);
        if (!done) {
          cst.wait(cst.cs, cst.mainfree()[b]);
          cst.copy(dkv_at(j, 0, g0), dkw, nkv * chunk_elems * 4);
          cst.copy(dkv_at(j, 1, g0), dkw + nkv * chunk_elems, nkv * chunk_elems * 4);
        }
      }
      Head2SeqDesc qb;  // row-major fp32 dQ -> bf16
      qb.src = dq; qb.src_f32 = true;
      qb.dst = seq; qb.ld_dst = ld_dseq; qb.S = Sc; qb.D = d; qb.n_heads = U;
      for (int k = 0; k <= U; ++k) qb.first[k] = static_cast<uint16_t>(k);
      for (int k = 0; k < U; ++k) {
        qb.dst_head[k] = static_cast<uint16_t>(k);
        qb.src_slot[k] = static_cast<uint16_t>(k);
      }
      L.h2s(qb);
      // dX rows of the chunk (+)= dQKV W_qkv[:, heads]^T ; dW_qkv[:, heads] += X_chunk^T dQKV
      std::vector<int> wheads(g.q_heads.begin(), g.q_heads.end());
      if (final_here)
        for (int part = 0; part < 2; ++part)
          for (int m = 0; m < nkv; ++m) wheads.push_back((part == 0 ? H : H + G) + g.kv_proj[m]);
      GemmDesc gx;
      gx.A = seq; gx.lda = ld_dseq; gx.a_rows = Sc; gx.a_cols = ld_dseq; gx.a_mn = false;
      gx.B = W_qkv; gx.ldb = qkv_ld; gx.b_rows = d_model; gx.b_cols = qkv_ld; gx.b_mn = false;
      gx.M = Sc; gx.N = d_model; gx.K = n_out * d;
      head_blocks(gx.bmap_k, wheads, d);
      upipe_bf16* dXc = dX + row0 * d_model;
      if (n_st == 1) {
        gx.out = dXc; gx.ldo = d_model; gx.out_mode = kOutBf16;
      } else if (dx_done == 0) {
        gx.out = dx32; gx.ldo = d_model; gx.out_mode = kOutF32;
      } else if (dx_done + 1 < n_st) {
        gx.out = dx32; gx.ldo = d_model; gx.out_mode = kOutF32Acc;
      } else {
        gx.out = dXc; gx.ldo = d_model; gx.out_mode = kOutBf16PlusF32; gx.aux = dx32; gx.ld_aux = d_model;
      }
      ++dx_done;
      L.gemm(gx);
      GemmDesc gw;
      gw.A = X + row0 * d_model; gw.lda = d_model; gw.a_rows = Sc; gw.a_cols = d_model; gw.a_mn = true;
      gw.B = seq; gw.ldb = ld_dseq; gw.b_rows = Sc; gw.b_cols = ld_dseq; gw.b_mn = true;
      gw.M = d_model; gw.N = n_out * d; gw.K = Sc;
      head_blocks(gw.omap_n, wheads, d);
      gw.out = dW_qkv; gw.ldo = qkv_ld; gw.out_mode = kOutF32Red;
      gw.split_k = choose_split_k(gw);
      L.gemm(gw);
    }
  }
  // dW_o = O_saved^T dY
  GemmDesc gwo;
  gwo.A = O_saved; gwo.lda = static_cast<long long>(H) * d; gwo.a_rows = S; gwo.a_cols = gwo.lda; gwo.a_mn = true;
  gwo.B = dY; gwo.ldb = d_model; gwo.b_rows = S; gwo.b_cols = d_model; gwo.b_mn = true;
  gwo.M = H * d; gwo.N = d_model; gwo.K = S;
  gwo.out = dW_o; gwo.ldo = d_model;
  gwo.split_k = choose_split_k(gwo);
  if (gwo.split_k > 1) {
    if (L.ok() && cudaMemsetAsync(dW_o, 0, static_cast<size_t>(H) * d * d_model * 4, L.st) != cudaSuccess)
      L.err = cudaErrorUnknown;
    gwo.out_mode = kOutF32Red;
  } else {
    gwo.out_mode = kOutF32;
  }
  L.gemm(gwo);
  return chunk_finish(L, cst, c, stats);
}
