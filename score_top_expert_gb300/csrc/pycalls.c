/*
 * CPython entry points for the router's hot calls: argument conversion only.
 *
 * Each function takes the arguments of the C entry point of the same name
 * (include/moe_router.h) as Python integers and floats -- device pointers as
 * integers, 0 for NULL, the stream as its raw handle -- converts them, calls
 * the library and returns its status code.  The Python binding uses these
 * instead of ctypes where the module was built: for decode-sized calls the
 * host cost of converting fourteen arguments through ctypes is a large part
 * of the latency.  Nothing here computes anything on the router's data.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <stdint.h>

#include "moe_router.h"

/* Convert args[0 .. n-1] by the format string: 'p' pointer (unsigned
 * integer), 'i' int, 'f' float.  Returns 0 on success, -1 with a Python
 * exception set. */
static int convert(PyObject* const* args, Py_ssize_t nargs, const char* fmt, void** out) {
  const Py_ssize_t n = (Py_ssize_t)strlen(fmt);
  if (nargs != n) {
    PyErr_Format(PyExc_TypeError, "expected %zd arguments, got %zd", n, nargs);
    return -1;
  }
  for (Py_ssize_t i = 0; i < n; ++i) {
    if (fmt[i] == 'p') {
      const unsigned long long v = PyLong_AsUnsignedLongLong(args[i]);
      if (v == (unsigned long long)-1 && PyErr_Occurred()) return -1;
      *(uintptr_t*)out[i] = (uintptr_t)v;
    } else if (fmt[i] == 'i') {
      const long v = PyLong_AsLong(args[i]);
      if (v == -1 && PyErr_Occurred()) return -1;
      if (v < INT32_MIN || v > INT32_MAX) {
        PyErr_SetString(PyExc_OverflowError, "integer argument out of int range");
        return -1;
      }
      *(int*)out[i] = (int)v;
    } else {
      const double v = PyFloat_AsDouble(args[i]);
      if (v == -1.0 && PyErr_Occurred()) return -1;
      *(float*)out[i] = (float)v;
    }
  }
  return 0;
}

static PyObject* call_topk_fwd(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
  uintptr_t logits, bias, probs, map, scores, stream;
  int dt, T, E, K, sf, ng, gk;
  float c;
  void* out[] = {&logits, &dt, &T, &E, &K, &sf, &ng, &gk, &c, &bias, &probs, &map, &scores,
                 &stream};
  if (convert(args, nargs, "piiiiiiifppppp", out) != 0) return NULL;
  const int rc = router_topk_fwd((const void*)logits, (mr_dtype)dt, T, E, K, (mr_score_func)sf,
                                 ng, gk, c, (const float*)bias, (void*)probs, (uint8_t*)map,
                                 (float*)scores, (mr_stream_t)stream);
  return PyLong_FromLong(rc);
}

static PyObject* call_topk_bwd(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
  uintptr_t grad, map, scores, grad_logits, stream;
  int dt, T, E, K, sf;
  float c;
  void* out[] = {&grad, &map, &scores, &dt, &T, &E, &K, &sf, &c, &grad_logits, &stream};
  if (convert(args, nargs, "pppiiiiifpp", out) != 0) return NULL;
  const int rc = router_topk_bwd((const void*)grad, (const uint8_t*)map, (const float*)scores,
                                 (mr_dtype)dt, T, E, K, (mr_score_func)sf, c, (void*)grad_logits,
                                 (mr_stream_t)stream);
  return PyLong_FromLong(rc);
}

static PyObject* call_aux_scores_fwd(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
  uintptr_t logits, scores, map, inter, stream;
  int dt, T, E, K, sf;
  void* out[] = {&logits, &dt, &T, &E, &K, &sf, &scores, &map, &inter, &stream};
  if (convert(args, nargs, "piiiiipppp", out) != 0) return NULL;
  const int rc = router_aux_scores_fwd((const void*)logits, (mr_dtype)dt, T, E, K,
                                       (mr_score_func)sf, (float*)scores, (uint8_t*)map,
                                       (float*)inter, (mr_stream_t)stream);
  return PyLong_FromLong(rc);
}

static PyObject* call_aux_scores_bwd(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
  uintptr_t grad, saved, grad_logits, stream;
  int dt, T, E, K, sf;
  void* out[] = {&grad, &saved, &dt, &T, &E, &K, &sf, &grad_logits, &stream};
  if (convert(args, nargs, "ppiiiiipp", out) != 0) return NULL;
  const int rc = router_aux_scores_bwd((const float*)grad, (const float*)saved, (mr_dtype)dt, T,
                                       E, K, (mr_score_func)sf, (void*)grad_logits,
                                       (mr_stream_t)stream);
  return PyLong_FromLong(rc);
}

static PyMethodDef kMethods[] = {
    {"router_topk_fwd", (PyCFunction)(void (*)(void))call_topk_fwd, METH_FASTCALL,
     "router_topk_fwd(logits, dtype, T, E, K, score_func, num_groups, group_topk, "
     "scaling_factor, expert_bias, probs, routing_map, scores, stream) -> status"},
    {"router_topk_bwd", (PyCFunction)(void (*)(void))call_topk_bwd, METH_FASTCALL,
     "router_topk_bwd(grad_probs, routing_map, scores, dtype, T, E, K, score_func, "
     "scaling_factor, grad_logits, stream) -> status"},
    {"router_aux_scores_fwd", (PyCFunction)(void (*)(void))call_aux_scores_fwd, METH_FASTCALL,
     "router_aux_scores_fwd(logits, dtype, T, E, K, score_func, scores, routing_map, "
     "intermediate, stream) -> status"},
    {"router_aux_scores_bwd", (PyCFunction)(void (*)(void))call_aux_scores_bwd, METH_FASTCALL,
     "router_aux_scores_bwd(grad_scores, saved, dtype, T, E, K, score_func, grad_logits, "
     "stream) -> status"},
    {NULL, NULL, 0, NULL}};

static struct PyModuleDef kModule = {PyModuleDef_HEAD_INIT, "_pycalls",
                                     "CPython entry points of the router's hot calls.", -1,
                                     kMethods};

PyMODINIT_FUNC PyInit__pycalls(void) { return PyModule_Create(&kModule); }
