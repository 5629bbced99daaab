// Host-buffer execution of the MLP step (mx_mlp_pipeline_*).  A step's raw
// inputs come from host memory and its outputs go back to host memory.  The
// copies run on two streams of their own (host->device and device->host) and
// are ordered against the launches of the step through events, at the points
// the step exposes (mx::StepHooks): an input's copy for the next step may
// start as soon as this step's only reader of it (its quantizer, or the bias
// epilogue) has run, and an output's copy back starts as soon as its writer
// has run, while the next step's writer of that output waits for the copy.
// So host traffic in both directions overlaps the kernels and each other,
// within a step and across consecutive steps, with one device buffer per
// tensor.  No device memory is allocated here: the caller owns every device
// buffer (as for mx_mlp_fwd_bwd) and every host buffer.
#include <cstdio>
#include <new>

#include "mx_internal.h"

struct mx_mlp_pipeline {
  mx_mlp_args_t dev;
  cudaStream_t compute = nullptr, copy_in = nullptr, copy_out = nullptr;
  cudaEvent_t in_ready[mx::T_COUNT] = {};   // input t is on the device
  cudaEvent_t in_free[mx::T_COUNT] = {};    // the step's reader of input t has run
  cudaEvent_t out_ready[mx::T_COUNT] = {};  // the step's writer of output t has run
  cudaEvent_t out_done[mx::T_COUNT] = {};   // output t is back in host memory
  cudaError_t err = cudaSuccess;            // first CUDA error seen while enqueuing
};

namespace {

struct TensorIO {
  void* dev;
  const void* host_in;
  void* host_out;
  size_t bytes;
};

// Device pointer and size of each tensor of the step (null: not used).
void step_tensors(const mx_mlp_args_t& a, const mx_mlp_host_io_t* io, TensorIO (&t)[mx::T_COUNT]) {
  const size_t R = (size_t)a.R, D = (size_t)a.D, F = (size_t)a.F, G = (size_t)a.G;
  const size_t F1 = a.act == MX_ACT_SWIGLU ? 2 * F : F;
  for (auto& x : t) x = TensorIO{nullptr, nullptr, nullptr, 0};
  auto in = [&](int k, const void* d, const void* h, size_t bytes) {
    if (d) t[k] = TensorIO{const_cast<void*>(d), h, nullptr, bytes};
  };
  auto out = [&](int k, void* d, void* h, size_t bytes) {
    if (d) t[k] = TensorIO{d, nullptr, h, bytes};
  };
  in(mx::T_X, a.x, io ? io->x : nullptr, R * D * 2);
  in(mx::T_W1, a.w1, io ? io->w1 : nullptr, G * F1 * D * 2);
  in(mx::T_W2, a.w2, io ? io->w2 : nullptr, G * D * F * 2);
  in(mx::T_DY, a.dy, io ? io->dy : nullptr, R * D * 2);
  if (a.act != MX_ACT_SWIGLU) {
    in(mx::T_B1, a.b1, io ? io->b1 : nullptr, F * 2);
    in(mx::T_B2, a.b2, io ? io->b2 : nullptr, D * 2);
    out(mx::T_DB1, a.db1, io ? io->db1 : nullptr, F * 4);
    out(mx::T_DB2, a.db2, io ? io->db2 : nullptr, D * 4);
  }
  out(mx::T_Y, a.y, io ? io->y : nullptr, R * D * 2);
  out(mx::T_DX, a.dx, io ? io->dx : nullptr, R * D * 2);
  out(mx::T_DW1, a.dw1, io ? io->dw1 : nullptr, G * F1 * D * 2);
  out(mx::T_DW2, a.dw2, io ? io->dw2 : nullptr, G * D * F * 2);
}

void note(mx_mlp_pipeline* p, cudaError_t e) {
  if (e != cudaSuccess && p->err == cudaSuccess) p->err = e;
}

void hook_before(void* ctx, int t) {
  auto* p = static_cast<mx_mlp_pipeline*>(ctx);
  if (mx::step_tensor_is_input(t)) note(p, cudaStreamWaitEvent(p->compute, p->in_ready[t], 0));
  else note(p, cudaStreamWaitEvent(p->compute, p->out_done[t], 0));
}

void hook_after(void* ctx, int t) {
  auto* p = static_cast<mx_mlp_pipeline*>(ctx);
  if (mx::step_tensor_is_input(t)) note(p, cudaEventRecord(p->in_free[t], p->compute));
  else note(p, cudaEventRecord(p->out_ready[t], p->compute));
}

mx_status_t cuda_error(cudaError_t e, const char* what) {
  char buf[256];
  snprintf(buf, sizeof(buf), "%s: %s", what, cudaGetErrorString(e));
  return mx::set_error(MX_ERR_CUDA, buf);
}

void release(mx_mlp_pipeline* p) {
  for (int k = 0; k < mx::T_COUNT; k++) {
    cudaEvent_t* ev[4] = {&p->in_ready[k], &p->in_free[k], &p->out_ready[k], &p->out_done[k]};
    for (cudaEvent_t* e : ev)
      if (*e) cudaEventDestroy(*e);
  }
  if (p->copy_in) cudaStreamDestroy(p->copy_in);
  if (p->copy_out) cudaStreamDestroy(p->copy_out);
  delete p;
}

}  // namespace

extern "C" {

mx_status_t mx_mlp_pipeline_create(const mx_mlp_args_t* dev, mx_stream_t stream, mx_mlp_pipeline_t** out) {
  if (out == nullptr) return mx::set_error(MX_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  mx_status_t st = mx::mlp_check(dev);
  if (st != MX_OK) return st;
  auto* p = new (std::nothrow) mx_mlp_pipeline();
  if (p == nullptr) return mx::set_error(MX_ERR_INVALID_ARG, "out of host memory");
  p->dev = *dev;
  p->compute = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamCreateWithFlags(&p->copy_in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->copy_out, cudaStreamNonBlocking);
  for (int k = 0; k < mx::T_COUNT && e == cudaSuccess; k++) {
    cudaEvent_t* ev[4] = {&p->in_ready[k], &p->in_free[k], &p->out_ready[k], &p->out_done[k]};
    for (cudaEvent_t* x : ev)
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(x, cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    release(p);
    return cuda_error(e, "pipeline streams and events");
  }
  *out = p;
  return MX_OK;
}

mx_status_t mx_mlp_pipeline_run(mx_mlp_pipeline_t* p, const mx_mlp_host_io_t* io) {
  if (p == nullptr || io == nullptr) return mx::set_error(MX_ERR_INVALID_ARG, "pipeline or io is NULL");
  if (p->err != cudaSuccess) return cuda_error(p->err, "an earlier pipeline step");
  const mx_mlp_args_t& a = p->dev;
  TensorIO t[mx::T_COUNT];
  step_tensors(a, io, t);
  // weights and their gradients may stay on the device (no host buffer)
  auto resident_ok = [](int k) { return k == mx::T_W1 || k == mx::T_W2 || k == mx::T_DW1 || k == mx::T_DW2; };
  for (int k = 0; k < mx::T_COUNT; k++) {
    if (t[k].dev == nullptr || resident_ok(k)) continue;
    if (mx::step_tensor_is_input(k) ? t[k].host_in == nullptr : t[k].host_out == nullptr) {
      char buf[96];
      snprintf(buf, sizeof(buf), "host buffer of step tensor %d is NULL", k);
      return mx::set_error(MX_ERR_INVALID_ARG, buf);
    }
  }
  if (a.offsets != nullptr && io->offsets == nullptr)
    return mx::set_error(MX_ERR_INVALID_ARG, "host offsets are NULL");
  if (a.R == 0) return MX_OK;
  // host -> device, in the order the step reads them
  const int in_order[] = {mx::T_X, mx::T_W1, mx::T_W2, mx::T_B1, mx::T_B2, mx::T_DY};
  for (int k : in_order) {
    if (t[k].dev == nullptr || t[k].host_in == nullptr) continue;
    note(p, cudaStreamWaitEvent(p->copy_in, p->in_free[k], 0));
    note(p, cudaMemcpyAsync(t[k].dev, t[k].host_in, t[k].bytes, cudaMemcpyHostToDevice, p->copy_in));
    note(p, cudaEventRecord(p->in_ready[k], p->copy_in));
  }
  // the routing (G int32) travels on the compute stream, behind the previous
  // step's last reader of it
  if (a.offsets != nullptr)
    note(p, cudaMemcpyAsync(const_cast<int32_t*>(a.offsets), io->offsets, (size_t)a.G * sizeof(int32_t),
                            cudaMemcpyHostToDevice, p->compute));
  if (p->err != cudaSuccess) return cuda_error(p->err, "pipeline copy-in");
  const mx::StepHooks hooks{hook_before, hook_after, p};
  mx_status_t st = mx::mlp_step(&a, reinterpret_cast<mx_stream_t>(p->compute), &hooks);
  if (st != MX_OK) return st;
  // device -> host, in the order the step writes them
  const int out_order[] = {mx::T_Y, mx::T_DB2, mx::T_DB1, mx::T_DX, mx::T_DW2, mx::T_DW1};
  for (int k : out_order) {
    if (t[k].dev == nullptr || t[k].host_out == nullptr) continue;
    note(p, cudaStreamWaitEvent(p->copy_out, p->out_ready[k], 0));
    note(p, cudaMemcpyAsync(t[k].host_out, t[k].dev, t[k].bytes, cudaMemcpyDeviceToHost, p->copy_out));
    note(p, cudaEventRecord(p->out_done[k], p->copy_out));
  }
  if (p->err != cudaSuccess) return cuda_error(p->err, "pipeline step");
  return MX_OK;
}

mx_status_t mx_mlp_pipeline_sync(mx_mlp_pipeline_t* p) {
  if (p == nullptr) return mx::set_error(MX_ERR_INVALID_ARG, "pipeline is NULL");
  note(p, cudaStreamSynchronize(p->copy_in));
  note(p, cudaStreamSynchronize(p->compute));
  note(p, cudaStreamSynchronize(p->copy_out));
  if (p->err != cudaSuccess) return cuda_error(p->err, "pipeline");
  return MX_OK;
}

void mx_mlp_pipeline_destroy(mx_mlp_pipeline_t* p) {
  if (p == nullptr) return;
  cudaStreamSynchronize(p->copy_in);
  cudaStreamSynchronize(p->compute);
  cudaStreamSynchronize(p->copy_out);
  release(p);
}

}  // extern "C"
