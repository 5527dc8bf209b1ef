// The Muon step on matrices whose parameters, gradients and momentum stay in
// host memory.
//
// Source: "Training a 1T-Parameter MoE on EU public infrastructure with
// PyTorch and TorchTitan", section "FlexShard: Muon without communication":
// with FSDP's CPU offload the optimizer state and parameters live in Grace
// memory, and running Newton-Schulz on the GPU while the parameters stay
// offloaded cut the optimizer step from 41.7 s to 2.2 s.
//
// Design: the batch is cut into chunks of `chunk` matrices that rotate through
// three device slots.  For chunk k (slot k % 3):
//   copy-in stream   waits until the slot's previous chunk has been copied out,
//                    then copies gradients, momentum and parameters in;
//   caller's stream  waits for the copy-in, runs the fused step (momentum ->
//                    Newton-Schulz -> update, muon_step_batched) on the slot;
//   copy-out stream  waits for the compute, copies parameters and momentum out.
// Copies of chunk k+1 and k-1 therefore overlap the compute of chunk k.  The
// host link, not the compute, bounds the call, so the copy-in stream must
// never wait: with two slots it waited for chunk k-2's copy-out before chunk
// k's copy-in, idling the link once per two chunks; a third slot gives the
// copy-out a chunk's time of slack (3.5-5.6% faster, back to back; the link's
// speed drifts between runs on a shared host).  The
// caller's stream finally waits for the last copy-out, so completion of the
// call on that stream means the host arrays hold the result.  Device memory
// (three slots and one Newton-Schulz workspace) is allocated and freed
// stream-ordered on the caller's stream.
#include <algorithm>

#include "common.cuh"

namespace muon {
namespace {

bool is_host_accessible_pinned(const void *p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

// The side streams and every event the call records, all created before any
// device memory is allocated, so that no failure after the allocation can
// skip the join of the side streams or the stream-ordered free.
constexpr int kSlots = 3;   // device slots the chunks rotate through

struct Streams {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t in_done[kSlots] = {}, compute_done[kSlots] = {}, out_done[kSlots] = {};
  cudaEvent_t ready = nullptr, tail[2] = {};
  ~Streams() {
    for (int i = 0; i < kSlots; ++i) {
      if (in_done[i]) cudaEventDestroy(in_done[i]);
      if (compute_done[i]) cudaEventDestroy(compute_done[i]);
      if (out_done[i]) cudaEventDestroy(out_done[i]);
    }
    for (int i = 0; i < 2; ++i)
      if (tail[i]) cudaEventDestroy(tail[i]);
    if (ready) cudaEventDestroy(ready);
    if (in) cudaStreamDestroy(in);    // deferred by CUDA until the enqueued work is done
    if (out) cudaStreamDestroy(out);
  }
  bool create() {
    if (cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&ready, cudaEventDisableTiming) != cudaSuccess) return false;
    for (int i = 0; i < kSlots; ++i)
      if (cudaEventCreateWithFlags(&in_done[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&compute_done[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&out_done[i], cudaEventDisableTiming) != cudaSuccess)
        return false;
    for (int i = 0; i < 2; ++i)
      if (cudaEventCreateWithFlags(&tail[i], cudaEventDisableTiming) != cudaSuccess) return false;
    return true;
  }
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace muon

using namespace muon;

namespace {

// Group g's chunk size: `chunk` matrices (0: 8), at most its batch.
int64_t chunk_of(const muon_host_group &g, int64_t chunk) {
  return chunk > 0 ? std::min(chunk, g.batch) : std::min<int64_t>(g.batch, 8);
}

// The checks of one group, without any launch (the pinned-memory query is the
// only CUDA call).
int check_group(const muon_host_group &g) {
  if (g.batch < 0 || g.rows < 1 || g.cols < 1) return MUON_ERR_INVALID_ARG;
  if (g.batch == 0) return MUON_OK;
  if (!g.param_host || !g.grad_host || !g.momentum_host) return MUON_ERR_INVALID_ARG;
  if (g.rows % 8 || g.cols % 8) return MUON_ERR_UNSUPPORTED;
  if (!is_host_accessible_pinned(g.param_host) || !is_host_accessible_pinned(g.grad_host) ||
      !is_host_accessible_pinned(g.momentum_host))
    return MUON_ERR_UNSUPPORTED;  // pageable host memory would serialise every copy
  return MUON_OK;
}

}  // namespace

extern "C" int muon_step_host_grouped(const muon_host_group *groups, int ngroups, float mu, int nesterov, int steps,
                                      const float coeffs[3], float eps, float lr, float weight_decay, int64_t chunk,
                                      muon_stream_t stream) {
  if (ngroups < 0 || (ngroups > 0 && !groups) || chunk < 0 || steps < 0 || !coeffs) return MUON_ERR_INVALID_ARG;
  // slots and workspace for the largest chunk of any group
  int64_t slot_elems = 0;
  size_t ws = 0;
  for (int i = 0; i < ngroups; ++i) {
    const int c = check_group(groups[i]);
    if (c != MUON_OK) return c;
    if (groups[i].batch == 0) continue;
    const int64_t ch = chunk_of(groups[i], chunk);
    slot_elems = std::max(slot_elems, ch * groups[i].rows * groups[i].cols);
    ws = std::max(ws, muon_step_workspace_bytes(ch, groups[i].rows, groups[i].cols));
  }
  if (slot_elems == 0) return MUON_OK;
  const size_t g_bytes = align256((size_t)slot_elems * 2), m_bytes = align256((size_t)slot_elems * 4);
  const size_t slot_bytes = 2 * g_bytes + m_bytes;  // grad, param (bf16) + momentum (fp32)
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  Streams st;
  if (!st.create()) {
    cudaGetLastError();
    return MUON_ERR_CUDA;
  }
  uint8_t *dev = nullptr;
  if (alloc_async(reinterpret_cast<void **>(&dev), kSlots * slot_bytes + ws, s) != cudaSuccess || !dev) {
    cudaGetLastError();
    return MUON_ERR_NO_MEMORY;
  }
  int status = MUON_OK;
  // the side streams must not touch the slots before the allocation is ordered
  if (cudaEventRecord(st.ready, s) != cudaSuccess || cudaStreamWaitEvent(st.in, st.ready, 0) != cudaSuccess ||
      cudaStreamWaitEvent(st.out, st.ready, 0) != cudaSuccess)
    status = MUON_ERR_CUDA;

  bool used[kSlots] = {};
  int64_t k = 0;  // chunks issued so far, over all groups: chunk k uses slot k % kSlots
  for (int gi = 0; gi < ngroups && status == MUON_OK; ++gi) {
    const muon_host_group &g = groups[gi];
    if (g.batch == 0) continue;
    const int64_t per = g.rows * g.cols, ch = chunk_of(g, chunk);
    auto *ph = static_cast<uint8_t *>(g.param_host);
    auto *gh = static_cast<const uint8_t *>(g.grad_host);
    auto *mh = reinterpret_cast<uint8_t *>(g.momentum_host);
    for (int64_t b0 = 0; b0 < g.batch && status == MUON_OK; b0 += ch, ++k) {
      const int slot = (int)(k % kSlots);
      const int64_t nb = std::min(ch, g.batch - b0);
      uint8_t *base = dev + slot * slot_bytes;
      auto *g_d = base, *p_d = base + g_bytes;
      auto *m_d = reinterpret_cast<float *>(base + 2 * g_bytes);
      const size_t gb = (size_t)nb * per * 2, mb = (size_t)nb * per * 4;
      const size_t go = (size_t)b0 * per * 2, mo = (size_t)b0 * per * 4;
      // copy in (after this slot's previous chunk has been copied out)
      if (used[slot]) cudaStreamWaitEvent(st.in, st.out_done[slot], 0);
      if (cudaMemcpyAsync(g_d, gh + go, gb, cudaMemcpyHostToDevice, st.in) != cudaSuccess ||
          cudaMemcpyAsync(m_d, mh + mo, mb, cudaMemcpyHostToDevice, st.in) != cudaSuccess ||
          cudaMemcpyAsync(p_d, ph + go, gb, cudaMemcpyHostToDevice, st.in) != cudaSuccess ||
          cudaEventRecord(st.in_done[slot], st.in) != cudaSuccess) {
        status = MUON_ERR_CUDA;
        break;
      }
      // compute on the caller's stream
      cudaStreamWaitEvent(s, st.in_done[slot], 0);
      status = muon_step_batched(p_d, g_d, m_d, nb, g.rows, g.cols, mu, nesterov, steps, coeffs, eps, lr,
                                 weight_decay, g.scale, dev + kSlots * slot_bytes, ws, stream);
      if (status != MUON_OK) break;
      cudaEventRecord(st.compute_done[slot], s);
      // copy out
      cudaStreamWaitEvent(st.out, st.compute_done[slot], 0);
      if (cudaMemcpyAsync(ph + go, p_d, gb, cudaMemcpyDeviceToHost, st.out) != cudaSuccess ||
          cudaMemcpyAsync(mh + mo, m_d, mb, cudaMemcpyDeviceToHost, st.out) != cudaSuccess ||
          cudaEventRecord(st.out_done[slot], st.out) != cudaSuccess) {
        status = MUON_ERR_CUDA;
        break;
      }
      used[slot] = true;
    }
  }
  // the caller's stream waits for all work on both side streams (also after an
  // error, when a copy may still be in flight), then releases the device memory
  cudaStream_t side[2] = {st.in, st.out};
  for (int i = 0; i < 2; ++i)
    if ((cudaEventRecord(st.tail[i], side[i]) != cudaSuccess || cudaStreamWaitEvent(s, st.tail[i], 0) != cudaSuccess) &&
        status == MUON_OK)
      status = MUON_ERR_CUDA;
  if (cudaFreeAsync(dev, s) != cudaSuccess && status == MUON_OK) status = MUON_ERR_CUDA;
  if (status == MUON_OK && cudaGetLastError() != cudaSuccess) status = MUON_ERR_CUDA;
  return status;
}

extern "C" int muon_step_host(void *param_host, const void *grad_host, float *momentum_host, int64_t batch,
                              int64_t rows, int64_t cols, float mu, int nesterov, int steps, const float coeffs[3],
                              float eps, float lr, float weight_decay, float scale, int64_t chunk,
                              muon_stream_t stream) {
  const muon_host_group g{param_host, grad_host, momentum_host, batch, rows, cols, scale};
  return muon_step_host_grouped(&g, 1, mu, nesterov, steps, coeffs, eps, lr, weight_decay, chunk, stream);
}
