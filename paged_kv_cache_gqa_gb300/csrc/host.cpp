// Host-side entry points of libmtkv: error reporting, row widths, move
// ordering and validation, the grow-on-demand capacity rule, and reading the
// device status word. No device memory is allocated anywhere in the library.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace mtkv {

static thread_local std::string g_last_error;

mt_status fail(mt_status st, const std::string &msg) {
  g_last_error = msg;
  return st;
}

mt_status ok() {
  g_last_error.clear();
  return MT_OK;
}

mt_status cuda_check(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return MT_OK;
  return fail(MT_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

mt_status kernel_smem(const void *kern, int bytes, const char *what, bool max_carveout) {
  static std::mutex mu;
  static std::map<std::pair<int, const void *>, int> done;  // (device, kernel) -> bytes set
  int dev = 0;
  mt_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != MT_OK) return st;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(dev, kern);
  const auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return MT_OK;
  st = cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                  what);
  if (st != MT_OK) return st;
  if (max_carveout) {
    st = cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared),
                    what);
    if (st != MT_OK) return st;
  }
  done[key] = bytes;
  return MT_OK;
}

mt_status device_info(DeviceInfo *out) {
  static std::mutex mu;
  static std::vector<DeviceInfo> cache;
  int dev = 0;
  mt_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != MT_OK) return st;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto &d : cache)
    if (d.device == dev) {
      *out = d;
      return MT_OK;
    }
  DeviceInfo d{dev, 0, 0};
  st = cuda_check(cudaDeviceGetAttribute(&d.n_sm, cudaDevAttrMultiProcessorCount, dev),
                  "cudaDeviceGetAttribute(SM count)");
  if (st != MT_OK) return st;
  st = cuda_check(cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev),
                  "cudaDeviceGetAttribute(shared memory)");
  if (st != MT_OK) return st;
  cache.push_back(d);
  *out = d;
  return MT_OK;
}

}  // namespace mtkv

using namespace mtkv;

extern "C" {

const char *mt_last_error(void) { return g_last_error.c_str(); }

const char *mt_version(void) { return "mtkv 0.1 (sm_103a)"; }

size_t mt_kv_row_bytes(mt_kv_format fmt, int n_kv_heads, int head_dim) {
  if (n_kv_heads <= 0 || head_dim <= 0) return 0;
  const size_t n = (size_t)n_kv_heads * (size_t)head_dim;
  switch (fmt) {
    case MT_KV_F32:
      return 4 * n;
    case MT_KV_F16:
      return 2 * n;
    case MT_KV_Q8_0: {
      if (head_dim % 32) return 0;
      const size_t raw = (n / 32) * 34;
      return (raw + 3) / 4 * 4;
    }
  }
  return 0;
}

mt_status mt_order_moves(mt_move *moves, int n_moves, int *n_out) {
  if (n_moves < 0 || (n_moves > 0 && !moves) || !n_out)
    return fail(MT_ERR_INVALID_ARG, "mt_order_moves: bad arguments");
  std::vector<mt_move> up, down;
  for (int i = 0; i < n_moves; ++i) {
    const mt_move &m = moves[i];
    if (m.len <= 0 || m.dst == m.src) continue;
    (m.dst > m.src ? up : down).push_back(m);
  }
  // upward moves top-down (source descending), then downward bottom-up
  std::stable_sort(up.begin(), up.end(),
                   [](const mt_move &a, const mt_move &b) { return a.src > b.src; });
  std::stable_sort(down.begin(), down.end(),
                   [](const mt_move &a, const mt_move &b) { return a.src < b.src; });
  int k = 0;
  for (const auto &m : up) moves[k++] = m;
  for (const auto &m : down) moves[k++] = m;
  *n_out = k;
  return ok();
}

mt_status mt_check_moves(const mt_move *moves, int n_moves, int64_t n_cells, int *first_bad) {
  if (first_bad) *first_bad = -1;
  if (n_moves < 0 || (n_moves > 0 && !moves) || n_cells < 0)
    return fail(MT_ERR_INVALID_ARG, "mt_check_moves: bad arguments");
  for (int i = 0; i < n_moves; ++i) {
    const mt_move &m = moves[i];
    if (m.len < 0 || m.src < 0 || m.dst < 0 || m.src + m.len > n_cells ||
        m.dst + m.len > n_cells) {
      if (first_bad) *first_bad = i;
      return fail(MT_ERR_INVALID_ARG, "mt_check_moves: move " + std::to_string(i) +
                                          " lies outside [0, n_cells)");
    }
  }
  // A move that writes a row some later move still has to read loses that
  // row's original content. Sweep: sort later sources by start and test each
  // destination against the sources of every later move.
  // (Quadratic in the worst case only for lists that are far from ordered;
  // ordered compactions keep the inner scan short.)
  struct Src {
    int64_t lo, hi;
    int idx;
  };
  std::vector<Src> srcs;
  srcs.reserve(n_moves);
  for (int i = 0; i < n_moves; ++i)
    if (moves[i].len > 0) srcs.push_back({moves[i].src, moves[i].src + moves[i].len, i});
  std::sort(srcs.begin(), srcs.end(), [](const Src &a, const Src &b) { return a.lo < b.lo; });
  // prefix max of source ends, to bound the scan
  std::vector<int64_t> max_hi(srcs.size());
  for (size_t k = 0; k < srcs.size(); ++k)
    max_hi[k] = std::max(srcs[k].hi, k ? max_hi[k - 1] : INT64_MIN);
  for (int i = 0; i < n_moves; ++i) {
    const mt_move &m = moves[i];
    if (m.len <= 0) continue;
    const int64_t w0 = m.dst, w1 = m.dst + m.len;
    // sources with lo < w1 and hi > w0 overlap the written range
    size_t k = std::lower_bound(srcs.begin(), srcs.end(), w1,
                                [](const Src &a, int64_t v) { return a.lo < v; }) -
               srcs.begin();
    while (k > 0) {
      --k;
      if (max_hi[k] <= w0) break;
      if (srcs[k].hi > w0 && srcs[k].idx > i) {
        if (first_bad) *first_bad = i;
        return fail(MT_ERR_ORDER, "mt_check_moves: move " + std::to_string(i) +
                                      " overwrites rows that move " +
                                      std::to_string(srcs[k].idx) + " has not copied yet");
      }
    }
  }
  return ok();
}

int64_t mt_kv_grow_capacity(int64_t cap, int64_t need, int64_t max_ctx) {
  if (cap <= 0 || max_ctx <= 0 || need < 0) return -1;
  int64_t nc = cap;
  while (nc < need) {
    if (nc > (INT64_MAX >> 1)) return -1;
    nc <<= 1;
  }
  return std::min(nc, max_ctx);
}

mt_status mt_check_device_status(uint32_t *status_word, mt_stream stream) {
  if (!status_word) return fail(MT_ERR_INVALID_ARG, "mt_check_device_status: null status word");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  mt_status st = cuda_check(cudaStreamSynchronize(s), "cudaStreamSynchronize");
  if (st != MT_OK) return st;
  st = cuda_check(cudaMemcpy(&v, status_word, sizeof(v), cudaMemcpyDeviceToHost),
                  "status read");
  if (st != MT_OK) return st;
  if (v) {
    st = cuda_check(cudaMemset(status_word, 0, sizeof(v)), "status clear");
    if (st != MT_OK) return st;
  }
  if (v & MT_STATUS_BIT_TIMEOUT)
    return fail(MT_ERR_TIMEOUT, "a bounded device-side wait ran out");
  if (v & MT_STATUS_BIT_DEVICE_CHECK)
    return fail(MT_ERR_DEVICE_CHECK,
                "a kernel skipped an out-of-range block id, context length or cell");
  return ok();
}

}  // extern "C"
