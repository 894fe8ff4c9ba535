// Packed per-layer block geometry.
//
// "MegaTrain" summary page, section on layer-contiguous memory tiling: each
// transformer layer's bf16 weights, bf16 gradients and fp32 Adam moments are
// packed into one contiguous block aligned to 4 KB pages, so one burst DMA
// moves the layer. The finer arrangement is this library's: segment-of-arrays
// (one segment per field), gradient first and written fields last, every
// tensor at an element index that is a multiple of 8, and the block's element
// count rounded up to 2048 so that every segment is a whole number of pages.
#include <cstring>
#include <new>

#include "lst_internal.h"

namespace lst {

const FormatInfo& format_info(lst_format fmt) {
  // field ids: G=0 W=1 M=2 V=3 MASTER=4
  static const FormatInfo l12 = {4, {0, 1, 2, 3, -1}, {2, 2, 4, 4, 0}, 4, 1, 12};
  static const FormatInfo l16m = {5, {0, 4, 2, 3, 1}, {2, 4, 4, 4, 2}, 4, 1, 16};
  static const FormatInfo l16f = {4, {0, 1, 2, 3, -1}, {4, 4, 4, 4, 0}, 4, 1, 16};
  switch (fmt) {
    case LST_L16_MIXED: return l16m;
    case LST_L16_FP32: return l16f;
    default: return l12;
  }
}

static int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

Run block_run(const lst_layout& L, const Block& b, char* base, int64_t e0, int64_t e1) {
  const FormatInfo& fi = format_info(L.fmt);
  auto seg = [&](int field) -> char* {
    int64_t off = b.seg_off[field];
    int es = 0;
    for (int k = 0; k < fi.n_segments; ++k)
      if (fi.field[k] == field) es = fi.elem_bytes[k];
    return base + off + e0 * es;
  };
  Run r;
  r.g = seg(LST_FIELD_G);
  r.m = reinterpret_cast<float*>(seg(LST_FIELD_M));
  r.v = reinterpret_cast<float*>(seg(LST_FIELD_V));
  if (L.fmt == LST_L16_MIXED) {
    r.w = seg(LST_FIELD_MASTER);
    r.w16 = seg(LST_FIELD_W);
  } else {
    r.w = seg(LST_FIELD_W);
    r.w16 = nullptr;
  }
  r.elems = e1 - e0;
  return r;
}

}  // namespace lst

using namespace lst;

extern "C" lst_status lst_layout_create(int32_t n_tensors, const int32_t* ndim, const int64_t* dims,
                                        const int32_t* layer_of_tensor, lst_format fmt,
                                        lst_layout** out) {
  clear_error();
  if (!out) return fail(LST_ERR_INVALID_ARG, "lst_layout_create: out is null");
  *out = nullptr;
  if (n_tensors < 0) return fail(LST_ERR_INVALID_ARG, "lst_layout_create: n_tensors < 0");
  if (n_tensors > 0 && (!ndim || !dims || !layer_of_tensor))
    return fail(LST_ERR_INVALID_ARG, "lst_layout_create: null shape arrays");
  if (fmt != LST_L12_BF16 && fmt != LST_L16_MIXED && fmt != LST_L16_FP32)
    return fail(LST_ERR_INVALID_ARG, "lst_layout_create: unknown format %d", (int)fmt);

  int64_t n_layers = 0;
  for (int32_t i = 0; i < n_tensors; ++i) {
    if (ndim[i] < 0 || ndim[i] > 4)
      return fail(LST_ERR_INVALID_ARG, "tensor %d: ndim %d outside 0..4", i, ndim[i]);
    if (layer_of_tensor[i] < 0)
      return fail(LST_ERR_INVALID_ARG, "tensor %d: negative block index", i);
    if (layer_of_tensor[i] + 1 > n_layers) n_layers = layer_of_tensor[i] + 1;
  }

  lst_layout* L = new (std::nothrow) lst_layout();
  if (!L) return fail(LST_ERR_OOM, "lst_layout_create: out of host memory");
  L->fmt = fmt;
  try {
    L->blocks.resize((size_t)n_layers);
    L->tensors.resize((size_t)n_tensors);
  } catch (...) {
    delete L;
    return fail(LST_ERR_OOM, "lst_layout_create: out of host memory");
  }
  std::vector<int64_t> cursor((size_t)n_layers, 0);
  std::vector<int64_t> count((size_t)n_layers, 0);
  for (int32_t i = 0; i < n_tensors; ++i) {
    int64_t n = 1;
    for (int k = 0; k < ndim[i]; ++k) {
      int64_t d = dims[4 * (int64_t)i + k];
      if (d < 0) {
        delete L;
        return fail(LST_ERR_INVALID_ARG, "tensor %d: negative dimension", i);
      }
      if (d != 0 && n > kMaxBlockElems / d) {
        delete L;
        return fail(LST_ERR_INVALID_ARG, "tensor %d: too many elements", i);
      }
      n *= d;
    }
    int64_t l = layer_of_tensor[i];
    Tensor& t = L->tensors[(size_t)i];
    t.layer = l;
    t.elem_off = cursor[(size_t)l];
    t.numel = n;
    cursor[(size_t)l] += round_up(n, kTensorAlign);
    if (cursor[(size_t)l] > kMaxBlockElems) {
      delete L;
      return fail(LST_ERR_INVALID_ARG, "block %lld larger than 2^40 elements", (long long)l);
    }
    L->blocks[(size_t)l].params += n;
    count[(size_t)l] += 1;
    L->n_params += n;
  }
  const FormatInfo& fi = format_info(fmt);
  for (int64_t l = 0; l < n_layers; ++l) {
    if (count[(size_t)l] == 0) {
      delete L;
      return fail(LST_ERR_INVALID_ARG, "block %lld has no tensors", (long long)l);
    }
    Block& b = L->blocks[(size_t)l];
    b.padded = round_up(cursor[(size_t)l], kBlockAlign);
    for (int f = 0; f < kMaxFields; ++f) b.seg_off[f] = -1;
    int64_t pos = 0;
    for (int k = 0; k < fi.n_segments; ++k) {
      b.seg_off[fi.field[k]] = pos;
      pos += b.padded * fi.elem_bytes[k];
    }
    b.bytes = pos;
    // inputs: segments [0, n_inputs); outputs: [first_output, n_segments)
    b.h2d_off = 0;
    b.h2d_bytes = 0;
    for (int k = 0; k < fi.n_inputs; ++k) b.h2d_bytes += b.padded * fi.elem_bytes[k];
    b.d2h_off = b.seg_off[fi.field[fi.first_output]];
    b.d2h_bytes = b.bytes - b.d2h_off;
    if (b.bytes > L->max_block_bytes) L->max_block_bytes = b.bytes;
  }
  *out = L;
  return LST_OK;
}

extern "C" void lst_layout_destroy(lst_layout* L) {
  if (!L) return;
  if (L->engine) destroy_engine(L->engine);
  delete L;
}

extern "C" lst_status lst_layout_info(const lst_layout* L, int64_t* n_layers, int64_t* n_params,
                                      int64_t* max_block_bytes) {
  clear_error();
  if (!L) return fail(LST_ERR_INVALID_ARG, "lst_layout_info: null layout");
  if (n_layers) *n_layers = (int64_t)L->blocks.size();
  if (n_params) *n_params = L->n_params;
  if (max_block_bytes) *max_block_bytes = L->max_block_bytes;
  return LST_OK;
}

extern "C" lst_status lst_layout_block(const lst_layout* L, int64_t layer, int64_t* bytes,
                                       int64_t* params, int64_t* padded_elems) {
  clear_error();
  if (!L) return fail(LST_ERR_INVALID_ARG, "lst_layout_block: null layout");
  if (layer < 0 || layer >= (int64_t)L->blocks.size())
    return fail(LST_ERR_INVALID_ARG, "lst_layout_block: block %lld out of range", (long long)layer);
  const Block& b = L->blocks[(size_t)layer];
  if (bytes) *bytes = b.bytes;
  if (params) *params = b.params;
  if (padded_elems) *padded_elems = b.padded;
  return LST_OK;
}

static int elem_bytes_of(lst_format fmt, int field) {
  const FormatInfo& fi = format_info(fmt);
  for (int k = 0; k < fi.n_segments; ++k)
    if (fi.field[k] == field) return fi.elem_bytes[k];
  return 0;
}

extern "C" lst_status lst_layout_segment(const lst_layout* L, int64_t layer, int32_t field,
                                         int64_t* byte_offset, int64_t* bytes) {
  clear_error();
  if (!L) return fail(LST_ERR_INVALID_ARG, "lst_layout_segment: null layout");
  if (layer < 0 || layer >= (int64_t)L->blocks.size())
    return fail(LST_ERR_INVALID_ARG, "lst_layout_segment: block %lld out of range", (long long)layer);
  if (field < 0 || field >= kMaxFields || elem_bytes_of(L->fmt, field) == 0)
    return fail(LST_ERR_INVALID_ARG, "lst_layout_segment: field %d not in this format", field);
  const Block& b = L->blocks[(size_t)layer];
  if (byte_offset) *byte_offset = b.seg_off[field];
  if (bytes) *bytes = b.padded * elem_bytes_of(L->fmt, field);
  return LST_OK;
}

extern "C" lst_status lst_layout_tensor(const lst_layout* L, int32_t tensor, int32_t field,
                                        int64_t* byte_offset, int64_t* layer, int64_t* elem_offset) {
  clear_error();
  if (!L) return fail(LST_ERR_INVALID_ARG, "lst_layout_tensor: null layout");
  if (tensor < 0 || tensor >= (int64_t)L->tensors.size())
    return fail(LST_ERR_INVALID_ARG, "lst_layout_tensor: tensor %d out of range", tensor);
  if (field < 0 || field >= kMaxFields || elem_bytes_of(L->fmt, field) == 0)
    return fail(LST_ERR_INVALID_ARG, "lst_layout_tensor: field %d not in this format", field);
  const Tensor& t = L->tensors[(size_t)tensor];
  const Block& b = L->blocks[(size_t)t.layer];
  if (byte_offset) *byte_offset = b.seg_off[field] + t.elem_off * elem_bytes_of(L->fmt, field);
  if (layer) *layer = t.layer;
  if (elem_offset) *elem_offset = t.elem_off;
  return LST_OK;
}

extern "C" lst_status lst_layout_transfer(const lst_layout* L, int64_t layer, int64_t* h2d_offset,
                                          int64_t* h2d_bytes, int64_t* d2h_offset, int64_t* d2h_bytes) {
  clear_error();
  if (!L) return fail(LST_ERR_INVALID_ARG, "lst_layout_transfer: null layout");
  if (layer < 0 || layer >= (int64_t)L->blocks.size())
    return fail(LST_ERR_INVALID_ARG, "lst_layout_transfer: block %lld out of range", (long long)layer);
  const Block& b = L->blocks[(size_t)layer];
  if (h2d_offset) *h2d_offset = b.h2d_off;
  if (h2d_bytes) *h2d_bytes = b.h2d_bytes;
  if (d2h_offset) *d2h_offset = b.d2h_off;
  if (d2h_bytes) *d2h_bytes = b.d2h_bytes;
  return LST_OK;
}

extern "C" lst_status lst_layout_set_stream_copy(lst_layout* L, int32_t h2d_mode, int32_t d2h_mode) {
  clear_error();
  if (!L) return fail(LST_ERR_INVALID_ARG, "lst_layout_set_stream_copy: null layout");
  auto ok = [](int32_t m) { return m == LST_COPY_ENGINE || m == LST_COPY_SM || m == LST_COPY_AUTO; };
  if (!ok(h2d_mode) || !ok(d2h_mode))
    return fail(LST_ERR_INVALID_ARG,
                "lst_layout_set_stream_copy: mode must be LST_COPY_ENGINE, LST_COPY_SM or LST_COPY_AUTO");
  std::lock_guard<std::mutex> g(L->stream_mu);
  L->stream_copy_h2d = h2d_mode;
  L->stream_copy_d2h = d2h_mode;
  L->link.clear();  // LST_COPY_AUTO measures again
  return LST_OK;
}

extern "C" lst_status lst_stream_copy_choice(const lst_layout* Lc, int64_t block, lst_copy_choice* out) {
  clear_error();
  if (!Lc || !out) return fail(LST_ERR_INVALID_ARG, "lst_stream_copy_choice: null argument");
  if (block < 0 || block >= (int64_t)Lc->blocks.size())
    return fail(LST_ERR_INVALID_ARG, "lst_stream_copy_choice: block %lld out of range", (long long)block);
  lst_layout* L = const_cast<lst_layout*>(Lc);  // the lock only
  std::lock_guard<std::mutex> g(L->stream_mu);
  lst_copy_choice c{};
  if ((size_t)block < L->link.size() && L->link[(size_t)block].measured) {
    const LinkChoice& k = L->link[(size_t)block];
    c.measured = 1;
    c.chunks = (int32_t)k.slow_in.size();
    for (size_t j = 0; j < k.slow_in.size(); ++j) {
      c.kernel_in_chunks += k.slow_in[j] ? 1 : 0;
      c.kernel_out_chunks += k.slow_out[j] ? 1 : 0;
    }
    c.engine_h2d_gbs_min = k.engine_h2d_min;
    c.engine_h2d_gbs_max = k.engine_h2d_max;
    c.engine_d2h_gbs_min = k.engine_d2h_min;
    c.engine_d2h_gbs_max = k.engine_d2h_max;
  }
  if (L->stream_copy_h2d != LST_COPY_AUTO) c.kernel_in_chunks = L->stream_copy_h2d == LST_COPY_SM ? c.chunks : 0;
  if (L->stream_copy_d2h != LST_COPY_AUTO) c.kernel_out_chunks = L->stream_copy_d2h == LST_COPY_SM ? c.chunks : 0;
  *out = c;
  return LST_OK;
}

extern "C" lst_status lst_layout_set_stream_chunk(lst_layout* L, int64_t elems) {
  clear_error();
  if (!L) return fail(LST_ERR_INVALID_ARG, "lst_layout_set_stream_chunk: null layout");
  if (elems < 0 || elems % kBlockAlign != 0)
    return fail(LST_ERR_INVALID_ARG, "stream chunk must be a non-negative multiple of 2048");
  std::lock_guard<std::mutex> g(L->stream_mu);
  L->stream_chunk = elems;
  return LST_OK;
}

extern "C" lst_status lst_stream_last_stats(const lst_layout* Lc, lst_stream_stats* out) {
  clear_error();
  if (!Lc || !out) return fail(LST_ERR_INVALID_ARG, "lst_stream_last_stats: null argument");
  lst_layout* L = const_cast<lst_layout*>(Lc);  // the lock only
  std::lock_guard<std::mutex> g(L->stream_mu);
  *out = L->last_step;
  return LST_OK;
}
