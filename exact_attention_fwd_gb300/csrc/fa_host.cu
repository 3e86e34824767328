// fa_host.cu — forward + backward on HOST buffers, pipelined over batch chunks.
//
// The batch is cut into chunks of up to `batch_chunk` sequences (every tensor
// is [B, ...] with B outermost, so a chunk is one contiguous slab per tensor);
// the first and last chunks are smaller (see ChunkPlan).
// Two device slots in the caller's workspace alternate: while chunk c is being
// computed, chunk c+1's inputs are copied in and chunk c-1's results copied
// out.  Three streams carry the work:
//   * an internal host-to-device copy stream: inputs of chunk c, after the
//     compute of chunk c-2 (same slot) has finished reading them;
//   * the caller's stream: fa_fwd then fa_bwd's phases on the slot, after its
//     inputs landed and chunk c-2's results have left the slot;
//   * an internal device-to-host copy stream: O, L, dQ, dK, dV of chunk c.
// The call orders all of it after the work already on the caller's stream,
// and the caller's stream waits for the last copies, so a stream
// synchronisation after the call covers every host write.  One
// cudaMemcpyAsync per tensor per chunk; the internal streams are created once
// per device and reused.
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "fa_common.cuh"

namespace {

constexpr int kMaxDevices = 64;
cudaStream_t g_copy_streams[kMaxDevices][2] = {};
std::mutex g_host_mu;   // also serialises the enqueue of concurrent calls

size_t elt_bytes(fa_dtype t) { return t == FA_DTYPE_F32 ? 4 : 2; }
size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Byte sizes of one slot's regions for a chunk of bc sequences.
struct SlotLayout {
  size_t in, grad, rows, ws;   // one input tensor, one gradient, one [bc,H,N] f32, bwd workspace
  size_t off_q, off_k, off_v, off_do, off_o, off_dq, off_dk, off_dv, off_lse, off_ws, total;
};

SlotLayout slot_layout(int bc, int H, int N, int d, fa_dtype dtype, fa_dtype grad_dtype) {
  SlotLayout s{};
  const size_t elems = static_cast<size_t>(bc) * N * H * d;
  s.in = elems * elt_bytes(dtype);
  s.grad = elems * elt_bytes(grad_dtype);
  s.rows = static_cast<size_t>(bc) * H * N * sizeof(float);
  s.ws = fa_bwd_workspace_size(bc, H, N);
  size_t o = 0;
  s.off_q = o;   o += up256(s.in);
  s.off_k = o;   o += up256(s.in);
  s.off_v = o;   o += up256(s.in);
  s.off_do = o;  o += up256(s.in);
  s.off_o = o;   o += up256(s.in);
  s.off_dq = o;  o += up256(s.grad);
  s.off_dk = o;  o += up256(s.grad);
  s.off_dv = o;  o += up256(s.grad);
  s.off_lse = o; o += up256(s.rows);
  s.off_ws = o;  o += up256(s.ws);
  s.total = o;
  return s;
}

fa_status copy_streams(cudaStream_t* h2d, cudaStream_t* d2h) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  for (int i = 0; i < 2; ++i)
    if (g_copy_streams[dev][i] == nullptr &&
        cudaStreamCreateWithFlags(&g_copy_streams[dev][i], cudaStreamNonBlocking) != cudaSuccess)
      return FA_ERR_CUDA;
  *h2d = g_copy_streams[dev][0];
  *d2h = g_copy_streams[dev][1];
  return FA_OK;
}

// Chunk sizes: bc/4 and bc/2 first, bc/2 and bc/4 last, full chunks between,
// so that the copy-in before the first kernels and the kernels and copy-out
// after the last copy-in (the parts nothing overlaps) are short.  Batches too
// small for the ramp use full chunks.
struct ChunkPlan {
  int bc, q, h, mid, nmid, n;   // mid: sequences in the full-size part
  bool ramp;
  ChunkPlan(int B, int bc_) : bc(bc_) {
    q = bc / 4 > 0 ? bc / 4 : 1;
    h = bc / 2 > 0 ? bc / 2 : 1;
    ramp = bc >= 4 && B >= 2 * (q + h) + bc;
    mid = ramp ? B - 2 * (q + h) : B;
    nmid = (mid + bc - 1) / bc;
    n = nmid + (ramp ? 4 : 0);
  }
  int size(int c) const {
    if (ramp) {
      if (c == 0 || c == n - 1) return q;
      if (c == 1 || c == n - 2) return h;
      c -= 2;
    }
    const int left = mid - c * bc;
    return left < bc ? left : bc;
  }
};

const char* cbyte(const void* p) { return static_cast<const char*>(p); }
char* byte(void* p) { return static_cast<char*>(p); }

}  // namespace

extern "C" {

size_t fa_fwd_bwd_host_workspace_size(int batch_chunk, int H, int N, int d, fa_dtype dtype,
                                      fa_dtype grad_dtype) {
  if (batch_chunk < 1 || H < 1 || N < 1 || d < 1) return 0;
  if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16) return 0;
  if (grad_dtype != dtype && grad_dtype != FA_DTYPE_F32) return 0;
  return 2 * slot_layout(batch_chunk, H, N, d, dtype, grad_dtype).total;
}

fa_status fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dO, void* o,
                          float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                          float scale, int causal, fa_dtype dtype, fa_dtype grad_dtype,
                          int batch_chunk, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (!q || !k || !v || !dO || !o || !lse || !dq || !dk || !dv || !workspace)
    return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16)
    return FA_ERR_INVALID_ARG;
  if (grad_dtype != dtype && grad_dtype != FA_DTYPE_F32) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1 || batch_chunk < 1) return FA_ERR_INVALID_ARG;
  if (d < 1 || d % 8 != 0 || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d > 128) return FA_ERR_UNSUPPORTED;
  const int bc = batch_chunk < B ? batch_chunk : B;
  const size_t need = fa_fwd_bwd_host_workspace_size(bc, H, N, d, dtype, grad_dtype);
  if (need == 0 || workspace_bytes < need) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return FA_ERR_INVALID_ARG;
  // the remaining size limits are fa_fwd's and fa_bwd's, checked per chunk

  const SlotLayout L = slot_layout(bc, H, N, d, dtype, grad_dtype);
  const size_t seq_in = static_cast<size_t>(N) * H * d * elt_bytes(dtype);   // one sequence
  const size_t seq_grad = static_cast<size_t>(N) * H * d * elt_bytes(grad_dtype);
  const size_t seq_rows = static_cast<size_t>(H) * N * sizeof(float);

  std::lock_guard<std::mutex> lock(g_host_mu);
  cudaStream_t cs = static_cast<cudaStream_t>(stream), hs = nullptr, ds = nullptr;
  fa_status st = copy_streams(&hs, &ds);
  if (st != FA_OK) return st;

  cudaEvent_t ev_start, ev_in[2], ev_done[2], ev_out[2];
  cudaEvent_t* all[] = {&ev_start, &ev_in[0], &ev_in[1], &ev_done[0], &ev_done[1],
                        &ev_out[0], &ev_out[1]};
  int made = 0;
  for (cudaEvent_t* e : all) {
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) {
      for (int i = 0; i < made; ++i) cudaEventDestroy(*all[i]);
      return FA_ERR_CUDA;
    }
    ++made;
  }
  auto ok = [&](cudaError_t e) {
    if (e != cudaSuccess && st == FA_OK) st = FA_ERR_CUDA;
    return st == FA_OK;
  };
  // everything after the work already queued on the caller's stream
  ok(cudaEventRecord(ev_start, cs));
  ok(cudaStreamWaitEvent(hs, ev_start, 0));
  ok(cudaStreamWaitEvent(ds, ev_start, 0));

  const ChunkPlan plan(B, bc);
  bool used[2] = {false, false};
  int b0 = 0;
  for (int c = 0; c < plan.n && st == FA_OK; b0 += plan.size(c), ++c) {
    const int s = c & 1;
    const int nb = plan.size(c);
    char* slot = byte(workspace) + static_cast<size_t>(s) * L.total;
    const size_t in_b = nb * seq_in, gr_b = nb * seq_grad, rw_b = nb * seq_rows;
    const size_t hin = static_cast<size_t>(b0) * seq_in, hgr = static_cast<size_t>(b0) * seq_grad,
                 hrw = static_cast<size_t>(b0) * seq_rows;
    // inputs in, once the slot's previous chunk has been computed
    if (used[s]) ok(cudaStreamWaitEvent(hs, ev_done[s], 0));
    ok(cudaMemcpyAsync(slot + L.off_q, cbyte(q) + hin, in_b, cudaMemcpyHostToDevice, hs));
    ok(cudaMemcpyAsync(slot + L.off_k, cbyte(k) + hin, in_b, cudaMemcpyHostToDevice, hs));
    ok(cudaMemcpyAsync(slot + L.off_v, cbyte(v) + hin, in_b, cudaMemcpyHostToDevice, hs));
    ok(cudaMemcpyAsync(slot + L.off_do, cbyte(dO) + hin, in_b, cudaMemcpyHostToDevice, hs));
    ok(cudaEventRecord(ev_in[s], hs));
    // compute on the caller's stream, once the slot's previous results left
    ok(cudaStreamWaitEvent(cs, ev_in[s], 0));
    if (used[s]) ok(cudaStreamWaitEvent(cs, ev_out[s], 0));
    if (st != FA_OK) break;
    float* lse_d = reinterpret_cast<float*>(slot + L.off_lse);
    st = fa_fwd(slot + L.off_q, slot + L.off_k, slot + L.off_v, slot + L.off_o, lse_d, nb, H, N,
                d, scale, causal, dtype, stream);
    if (st == FA_OK)
      st = fa_bwd(slot + L.off_q, slot + L.off_k, slot + L.off_v, slot + L.off_o, lse_d,
                  slot + L.off_do, slot + L.off_dq, slot + L.off_dk, slot + L.off_dv, nb, H, N, d,
                  scale, causal, dtype, grad_dtype, slot + L.off_ws, L.ws, stream);
    if (st != FA_OK) break;
    ok(cudaEventRecord(ev_done[s], cs));
    // results out
    ok(cudaStreamWaitEvent(ds, ev_done[s], 0));
    ok(cudaMemcpyAsync(byte(o) + hin, slot + L.off_o, in_b, cudaMemcpyDeviceToHost, ds));
    ok(cudaMemcpyAsync(reinterpret_cast<char*>(lse) + hrw, slot + L.off_lse, rw_b,
                       cudaMemcpyDeviceToHost, ds));
    ok(cudaMemcpyAsync(byte(dq) + hgr, slot + L.off_dq, gr_b, cudaMemcpyDeviceToHost, ds));
    ok(cudaMemcpyAsync(byte(dk) + hgr, slot + L.off_dk, gr_b, cudaMemcpyDeviceToHost, ds));
    ok(cudaMemcpyAsync(byte(dv) + hgr, slot + L.off_dv, gr_b, cudaMemcpyDeviceToHost, ds));
    ok(cudaEventRecord(ev_out[s], ds));
    used[s] = true;
  }
  // the caller's stream covers every copy of this call (also after a failure:
  // whatever was queued is waited for, so the slots are free again)
  ok(cudaEventRecord(ev_in[0], hs));
  ok(cudaEventRecord(ev_out[0], ds));
  cudaStreamWaitEvent(cs, ev_in[0], 0);
  cudaStreamWaitEvent(cs, ev_out[0], 0);
  for (cudaEvent_t* e : all) cudaEventDestroy(*e);   // released once they complete
  return st;
}

}  // extern "C"
