/*
 * CPython entry point for the prepared-layer call of libw4a16.so: converts the seven integer
 * arguments of w4a16_layer_gemm and calls it through a function pointer that the Python binding
 * resolves once from the library (ctypes) and hands over with bind(). Argument marshalling only:
 * no computation happens here. It exists because a ctypes call converts its arguments through
 * per-argument Python objects, which costs more host time per call than the small decode kernels
 * take on the GPU.
 *
 *   bind(address)                                    address of w4a16_layer_gemm
 *   layer_gemm(layer, a, out, m, ws, ws_bytes, stream) -> status (int)
 *     layer, a, out, ws, stream: integers (addresses; None or 0 for a null pointer);
 *     m: int64; ws_bytes: size_t. The GIL is released around the call.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <stddef.h>
#include <stdint.h>

typedef int (*layer_gemm_fn)(void *layer, const void *a, void *out, int64_t m, void *workspace,
                             size_t workspace_bytes, void *stream);
static layer_gemm_fn g_layer_gemm = NULL;

static void *as_ptr(PyObject *o) {
  if (o == Py_None) return NULL;
  return PyLong_AsVoidPtr(o);
}

static PyObject *bind(PyObject *self, PyObject *arg) {
  (void)self;
  void *p = PyLong_AsVoidPtr(arg);
  if (p == NULL) {
    if (!PyErr_Occurred()) PyErr_SetString(PyExc_ValueError, "bind: null function address");
    return NULL;
  }
  g_layer_gemm = (layer_gemm_fn)p;
  Py_RETURN_NONE;
}

static PyObject *layer_gemm(PyObject *self, PyObject *const *args, Py_ssize_t nargs) {
  (void)self;
  if (nargs != 7) {
    PyErr_SetString(PyExc_TypeError, "layer_gemm takes 7 arguments (layer, a, out, m, ws, ws_bytes, stream)");
    return NULL;
  }
  if (g_layer_gemm == NULL) {
    PyErr_SetString(PyExc_RuntimeError, "layer_gemm: bind() was not called");
    return NULL;
  }
  void *layer = as_ptr(args[0]);
  const void *a = as_ptr(args[1]);
  void *out = as_ptr(args[2]);
  const long long m = PyLong_AsLongLong(args[3]);
  void *ws = as_ptr(args[4]);
  const size_t ws_bytes = args[5] == Py_None ? 0 : PyLong_AsSize_t(args[5]);
  void *stream = as_ptr(args[6]);
  if (PyErr_Occurred()) return NULL;
  int st;
  Py_BEGIN_ALLOW_THREADS
  st = g_layer_gemm(layer, a, out, (int64_t)m, ws, ws_bytes, stream);
  Py_END_ALLOW_THREADS
  return PyLong_FromLong(st);
}

static PyMethodDef kMethods[] = {
    {"bind", (PyCFunction)bind, METH_O, "bind(address of w4a16_layer_gemm)"},
    {"layer_gemm", (PyCFunction)(void (*)(void))layer_gemm, METH_FASTCALL,
     "layer_gemm(layer, a, out, m, ws, ws_bytes, stream) -> status"},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef kModule = {PyModuleDef_HEAD_INIT, "_w4a16_call",
                                     "Argument marshalling for w4a16_layer_gemm.", -1, kMethods,
                                     NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__w4a16_call(void) { return PyModule_Create(&kModule); }
