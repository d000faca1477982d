// stack_api.cu -- the stacked-layer calls of the C ABI (prnn_stack_*): plan,
// weight packing and launch of the wavefront kernel, and the layer-by-layer
// comparison path built on single-layer handles.  Contracts are in
// include/prnn.h.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "host_util.h"
#include "prnn.h"
#include "prnn_internal.h"

using namespace prnn;

struct prnn_stack {
  int L = 0, H = 0, I = 0, maxB = 0;
  prnn_dtype_t wdtype = PRNN_F32;
  prnn_stack_algo_t algo = PRNN_STACK_WAVEFRONT;
  int device = 0, sm_count = 0;
  size_t smem_optin = 0;
  // wavefront plan (shared by every slice)
  int G = 1, cpg = 0, R = 0, n_cta = 0, nthreads = 0, cpt = 0, bw = 1;
  size_t smem = 0;
  int groups_opt = 0;
  std::vector<void*> Wpk;      // per layer: [cpg][cpt][R][nthreads] vec4
  std::vector<float*> bias;    // per layer [H]
  std::vector<char> set;       // per layer: weights present
  // layer-by-layer path
  std::vector<prnn_t> layer;
  int* status = nullptr;       // device int[4]
  long long timeout_us = 500000;
  int poll_delay_ns = kDenseDelayNs, clock_khz = 2000000;
  int backoff_ns = kStackBackoffNs;
  int drop_cta = -1, drop_step = -1, timing = 0;
  cudaEvent_t ev[2] = {nullptr, nullptr};
  bool ev_valid = false, sticky_timeout = false;
};

namespace {

// Wavefront plan: L slices of sm_count / L CTAs; each slice split into G
// groups of cpg CTAs with R rows each (R >= 5: the kernel's smallest row
// template is 8); threads cover the (I + H) / 4 chunks of the widest layer.
// Among the variants that fit (registers without spills, shared memory), the
// one with the least estimated step time: every batch pass costs one
// exchange round trip (~1.1 us on GB300) plus the larger of its FMA time and
// its shared-memory weight reads, at ~1.9 GHz.  A forced G keeps only that G.
bool plan_stack(prnn_stack* s) {
  const bool f16 = s->wdtype == PRNN_F16;
  const int per = s->sm_count / s->L;
  const int K = std::max(s->I, s->H) + s->H;
  const int nchunks = K / 4;
  const int gmax = s->groups_opt > 0 ? std::min(s->groups_opt, s->maxB) : std::min(s->maxB, 8);
  double best = 1e30;
  bool found = false;
  for (int G = gmax; G >= 1; --G) {
    if (s->groups_opt == 0 && G > 1 && (G & (G - 1)) != 0) continue;
    if (s->groups_opt > 0 && G != gmax) break;
    int cpg = per / G;
    if (cpg < 1) continue;
    const int R = std::max(5, (s->H + cpg - 1) / cpg);
    cpg = (s->H + R - 1) / R;
    const int rmax = recur_dense_rmax(R);
    if (rmax < 8) continue;
    const int bl = (s->maxB + G - 1) / G;
    for (int bw = recur_dense_bw(bl); bw >= 1; bw /= 2) {
      for (int cap : {512, 256}) {
        const int cpt = (nchunks + cap - 1) / cap;
        if (cpt > 4) continue;
        int nt = std::max(32, round_up((nchunks + cpt - 1) / cpt, 32));
        nt = std::max(nt, round_up(rmax * bw, 32));
        if (nt > dense_launch_bound(f16, rmax, bw, cpt)) continue;
        if (!stack_variant_ok(f16, rmax, bw, cpt)) continue;
        const size_t sm = recur_stack_smem(R, cpt, nt, f16, bw);
        if (sm > s->smem_optin) continue;
        const int passes = (bl + bw - 1) / bw;
        const double fma_ns = (double)R * K * bl / (128.0 * 1.9);
        const double smem_ns = (double)passes * R * K * (f16 ? 2 : 4) / (128.0 * 1.9);
        const double est = passes * 1100.0 + std::max(fma_ns, smem_ns);
        if (est < best) {
          best = est;
          found = true;
          s->G = G;
          s->cpg = cpg;
          s->R = R;
          s->n_cta = G * cpg;
          s->nthreads = nt;
          s->cpt = cpt;
          s->bw = bw;
          s->smem = sm;
        }
      }
    }
  }
  return found;
}

void free_layers(prnn_stack* s) {
  for (auto& p : s->Wpk) free_dev(p);
  for (auto& p : s->bias) free_dev(p);
  std::fill(s->set.begin(), s->set.end(), 0);
}

}  // namespace

extern "C" {

prnn_status_t prnn_stack_create(prnn_stack_t* out, int layers, int hidden, int input,
                                int max_batch, prnn_dtype_t wdtype, prnn_stack_algo_t algo) {
  if (!out) return PRNN_ERR_INVALID_ARG;
  *out = nullptr;
  if (layers < 1 || layers > kStackMaxLayers || hidden < 1 || input < 1 || max_batch < 1 ||
      max_batch > 32)
    return PRNN_ERR_INVALID_ARG;
  if (wdtype != PRNN_F32 && wdtype != PRNN_F16) return PRNN_ERR_INVALID_ARG;
  if (algo != PRNN_STACK_WAVEFRONT && algo != PRNN_STACK_LAYERWISE) return PRNN_ERR_INVALID_ARG;
  if (algo == PRNN_STACK_WAVEFRONT && (hidden % 4 != 0 || input % 4 != 0))
    return PRNN_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PRNN_ERR_UNSUPPORTED;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return PRNN_ERR_UNSUPPORTED;
  if (prop.major != 10 || prop.minor != 3 || !prop.cooperativeLaunch) return PRNN_ERR_UNSUPPORTED;
  prnn_stack* s = new (std::nothrow) prnn_stack();
  if (!s) return PRNN_ERR_OOM;
  s->L = layers;
  s->H = hidden;
  s->I = input;
  s->maxB = max_batch;
  s->wdtype = wdtype;
  s->algo = algo;
  s->device = dev;
  s->sm_count = prop.multiProcessorCount;
  s->smem_optin = prop.sharedMemPerBlockOptin;
  if (cudaDeviceGetAttribute(&s->clock_khz, cudaDevAttrClockRate, dev) != cudaSuccess)
    s->clock_khz = 2000000;
  s->Wpk.assign(layers, nullptr);
  s->bias.assign(layers, nullptr);
  s->set.assign(layers, 0);
  prnn_status_t st = PRNN_OK;
  if (algo == PRNN_STACK_WAVEFRONT && !plan_stack(s)) st = PRNN_ERR_UNSUPPORTED;
  if (st == PRNN_OK && algo == PRNN_STACK_LAYERWISE) {
    s->layer.assign(layers, nullptr);
    for (int l = 0; l < layers && st == PRNN_OK; ++l)
      st = prnn_create(&s->layer[l], hidden, l == 0 ? input : hidden, max_batch, wdtype,
                       PRNN_ALGO_PERSISTENT);
  }
  if (st == PRNN_OK && (cudaMalloc((void**)&s->status, 4 * sizeof(int)) != cudaSuccess ||
                        cudaMemset(s->status, 0, 4 * sizeof(int)) != cudaSuccess))
    st = PRNN_ERR_OOM;
  for (int i = 0; i < 2 && st == PRNN_OK; ++i)
    if (cudaEventCreate(&s->ev[i]) != cudaSuccess) st = PRNN_ERR_CUDA;
  if (st != PRNN_OK) {
    prnn_stack_destroy(s);
    return st;
  }
  *out = s;
  return PRNN_OK;
}

prnn_status_t prnn_stack_destroy(prnn_stack_t s) {
  if (!s) return PRNN_OK;
  cudaSetDevice(s->device);
  free_layers(s);
  for (prnn_t h : s->layer) prnn_destroy(h);
  free_dev(s->status);
  for (auto& e : s->ev)
    if (e) cudaEventDestroy(e);
  delete s;
  return PRNN_OK;
}

prnn_status_t prnn_stack_set_layer(prnn_stack_t s, int layer, const void* Wx, const void* Wh,
                                   const float* bias, void* stream) {
  if (!s || !Wx || !Wh || !bias || layer < 0 || layer >= s->L) return PRNN_ERR_INVALID_ARG;
  if (s->sticky_timeout) return PRNN_ERR_TIMEOUT;
  if (s->algo == PRNN_STACK_LAYERWISE)
    return prnn_set_weights_dense(s->layer[layer], Wx, Wh, bias, stream);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PRNN_TRY(cudaStreamSynchronize(st));
  const int H = s->H, I = layer == 0 ? s->I : s->H;
  const size_t esz = s->wdtype == PRNN_F16 ? 2 : 4;
  std::vector<unsigned char> wx((size_t)H * I * esz), wh((size_t)H * H * esz);
  std::vector<float> b((size_t)H);
  PRNN_TRY(to_host(wx.data(), Wx, wx.size()));
  PRNN_TRY(to_host(wh.data(), Wh, wh.size()));
  PRNN_TRY(to_host(b.data(), bias, b.size() * sizeof(float)));
  // per CTA of a group: [chunk slot j][row r][thread i] -> 4 weights of row
  // cta*R + r of [Wx | Wh], columns 4*(i + j*nthreads) .. +3 (zero outside)
  const int NT = s->nthreads, ic = I / 4, nchunks = ic + H / 4;
  const size_t vec = 4 * esz;
  std::vector<unsigned char> pk((size_t)s->cpg * s->cpt * s->R * NT * vec, 0);
  for (int cta = 0; cta < s->cpg; ++cta)
    for (int j = 0; j < s->cpt; ++j)
      for (int r = 0; r < s->R; ++r)
        for (int i = 0; i < NT; ++i) {
          const int row = cta * s->R + r, ch = i + j * NT;
          if (row >= H || ch >= nchunks) continue;
          const size_t dst = ((((size_t)cta * s->cpt + j) * s->R + r) * NT + i) * vec;
          const unsigned char* src = ch < ic
                                         ? &wx[((size_t)row * I + (size_t)ch * 4) * esz]
                                         : &wh[((size_t)row * H + (size_t)(ch - ic) * 4) * esz];
          std::memcpy(&pk[dst], src, vec);
        }
  free_dev(s->Wpk[layer]);
  free_dev(s->bias[layer]);
  s->set[layer] = 0;
  PRNN_TRY(upload(&s->Wpk[layer], pk.data(), pk.size()));
  PRNN_TRY(upload(&s->bias[layer], b.data(), b.size() * sizeof(float)));
  s->set[layer] = 1;
  return PRNN_OK;
}

prnn_status_t prnn_stack_forward(prnn_stack_t s, int T, int B, const float* x, const float* h0,
                                 float* y, void* stream) {
  if (!s) return PRNN_ERR_INVALID_ARG;
  if (s->sticky_timeout) return PRNN_ERR_TIMEOUT;
  if (T < 0 || B < 0 || B > s->maxB) return PRNN_ERR_INVALID_ARG;
  if (s->algo == PRNN_STACK_WAVEFRONT) {
    for (int l = 0; l < s->L; ++l)
      if (!s->set[l]) return PRNN_ERR_NOT_READY;
  } else {
    prnn_info_t info;
    for (prnn_t h : s->layer)
      if (prnn_get_info(h, &info) != PRNN_OK || !info.weights_set) return PRNN_ERR_NOT_READY;
  }
  if (T == 0 || B == 0) return PRNN_OK;
  if (!x || !y) return PRNN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || (h0 && !aligned16(h0))) return PRNN_ERR_INVALID_ARG;
  const size_t layer_y = (size_t)T * B * s->H;
  const size_t ny = layer_y * s->L;
  if (overlaps(y, ny * 4, x, (size_t)T * B * s->I * 4)) return PRNN_ERR_INVALID_ARG;
  if (h0 && overlaps(y, ny * 4, h0, (size_t)s->L * B * s->H * 4)) return PRNN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (s->timing) PRNN_TRY(cudaEventRecord(s->ev[0], st));

  if (s->algo == PRNN_STACK_LAYERWISE) {
    for (int l = 0; l < s->L; ++l) {
      const float* in = l == 0 ? x : y + (size_t)(l - 1) * layer_y;
      const float* h0l = h0 ? h0 + (size_t)l * B * s->H : nullptr;
      prnn_status_t r = prnn_forward(s->layer[l], T, B, in, h0l, y + (size_t)l * layer_y, stream);
      if (r != PRNN_OK) return r;
    }
  } else {
    PRNN_TRY(launch_fill_sentinel(y, ny, st));
    StackArgs a{};
    RecurCommon& c = a.c;
    c.T = T;
    c.B = B;
    c.H = s->H;
    c.n_cta = s->n_cta;
    c.R = s->R;
    c.G = s->G;
    c.cpg = s->cpg;
    c.nthreads = s->nthreads;
    c.smem = s->smem;
    c.status = s->status;
    c.timeout_ns = s->timeout_us * 1000LL;
    c.poll_delay = (int)((long long)s->poll_delay_ns * s->clock_khz / 1000000LL);
    c.poll_backoff = (int)((long long)s->backoff_ns * s->clock_khz / 1000000LL);
    c.drop_cta = s->drop_cta;
    c.drop_step = s->drop_step;
    a.L = s->L;
    a.cpt = s->cpt;
    a.wfp16 = s->wdtype == PRNN_F16;
    for (int l = 0; l < s->L; ++l) {
      StackLayerArgs& la = a.layer[l];
      la.Wpk = s->Wpk[l];
      la.bias = s->bias[l];
      la.xin = l == 0 ? x : y + (size_t)(l - 1) * layer_y;
      la.y = y + (size_t)l * layer_y;
      la.h0 = h0 ? h0 + (size_t)l * B * s->H : nullptr;
      la.I = l == 0 ? s->I : s->H;
      la.poll_in = l > 0;
    }
    PRNN_TRY(launch_recur_stack(a, s->bw, st));
  }
  if (s->timing) {
    PRNN_TRY(cudaEventRecord(s->ev[1], st));
    s->ev_valid = true;
  }
  return PRNN_OK;
}

prnn_status_t prnn_stack_get_status(prnn_stack_t s, void* stream) {
  if (!s) return PRNN_ERR_INVALID_ARG;
  PRNN_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  if (s->algo == PRNN_STACK_LAYERWISE) {
    for (prnn_t h : s->layer)
      if (prnn_get_status(h, nullptr) == PRNN_ERR_TIMEOUT) s->sticky_timeout = true;
  } else {
    int w[4] = {0, 0, 0, 0};
    PRNN_TRY(cudaMemcpy(w, s->status, sizeof(w), cudaMemcpyDeviceToHost));
    if (w[0] != 0) s->sticky_timeout = true;
  }
  return s->sticky_timeout ? PRNN_ERR_TIMEOUT : PRNN_OK;
}

prnn_status_t prnn_stack_set_option(prnn_stack_t s, prnn_option_t opt, long long value) {
  if (!s) return PRNN_ERR_INVALID_ARG;
  switch (opt) {
    case PRNN_OPT_WAIT_TIMEOUT_US:
      if (value < 1 || value > 60LL * 1000 * 1000) return PRNN_ERR_INVALID_ARG;
      s->timeout_us = value;
      for (prnn_t h : s->layer) prnn_set_option(h, opt, value);
      return PRNN_OK;
    case PRNN_OPT_POLL_DELAY_NS:
      if (value < 0 || value > 10000) return PRNN_ERR_INVALID_ARG;
      s->poll_delay_ns = (int)value;
      for (prnn_t h : s->layer) prnn_set_option(h, opt, value);
      return PRNN_OK;
    case PRNN_OPT_POLL_BACKOFF_NS:
      if (value < 0 || value > 10000) return PRNN_ERR_INVALID_ARG;
      s->backoff_ns = (int)value;
      for (prnn_t h : s->layer) prnn_set_option(h, opt, value);
      return PRNN_OK;
    case PRNN_OPT_TIMING:
      if (value != 0 && value != 1) return PRNN_ERR_INVALID_ARG;
      s->timing = (int)value;
      s->ev_valid = false;
      return PRNN_OK;
    case PRNN_OPT_DEBUG_DROP_CTA:
      if (value < -1 || value > 1 << 20) return PRNN_ERR_INVALID_ARG;
      s->drop_cta = (int)value;
      return PRNN_OK;
    case PRNN_OPT_DEBUG_DROP_STEP:
      if (value < -1 || value > 1 << 30) return PRNN_ERR_INVALID_ARG;
      s->drop_step = (int)value;
      return PRNN_OK;
    case PRNN_OPT_CTA_GROUPS: {
      if (s->algo != PRNN_STACK_WAVEFRONT || value < 0 || value > 32) return PRNN_ERR_INVALID_ARG;
      const int old = s->groups_opt;
      s->groups_opt = (int)value;
      if (!plan_stack(s)) {
        s->groups_opt = old;
        plan_stack(s);
        return PRNN_ERR_UNSUPPORTED;
      }
      free_layers(s);
      return PRNN_OK;
    }
    default:
      return PRNN_ERR_INVALID_ARG;
  }
}

prnn_status_t prnn_stack_get_timing(prnn_stack_t s, float* ms) {
  if (!s || !ms) return PRNN_ERR_INVALID_ARG;
  if (!s->timing || !s->ev_valid) return PRNN_ERR_NOT_READY;
  PRNN_TRY(cudaEventSynchronize(s->ev[1]));
  PRNN_TRY(cudaEventElapsedTime(ms, s->ev[0], s->ev[1]));
  return PRNN_OK;
}

prnn_status_t prnn_stack_get_info(prnn_stack_t s, prnn_stack_info_t* info) {
  if (!s || !info) return PRNN_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  info->layers = s->L;
  info->hidden = s->H;
  info->input = s->I;
  info->max_batch = s->maxB;
  info->wdtype = s->wdtype;
  info->algo = s->algo;
  int n = 0;
  if (s->algo == PRNN_STACK_WAVEFRONT) {
    for (char c : s->set) n += c ? 1 : 0;
    info->n_cta_per_layer = s->n_cta;
    info->rows_per_cta = s->R;
    info->threads_per_cta = s->nthreads;
    info->cta_groups = s->G;
    info->batch_per_pass = s->bw;
    info->chunks_per_thread = s->cpt;
    info->smem_bytes = (long long)s->smem;
    info->onchip_weight_bytes = (long long)s->L * s->n_cta * s->cpt * s->R * s->nthreads * 4 *
                                (s->wdtype == PRNN_F16 ? 2 : 4);
  } else {
    prnn_info_t li;
    for (prnn_t h : s->layer)
      if (prnn_get_info(h, &li) == PRNN_OK && li.weights_set) {
        ++n;
        info->onchip_weight_bytes = std::max(info->onchip_weight_bytes,
                                             (long long)li.onchip_weight_bytes);
      }
  }
  info->layers_set = n;
  return PRNN_OK;
}

}  // extern "C"
