/* _rxstep: the per-step argument marshalling of the engine's one-call step, as a CPython
 * extension.  It writes the step's inputs into a caller-owned rx_step_args / rx_step_io pair
 * and calls rx_step_run (whose address the binding passes in once, from the loaded library):
 * the same call the ctypes binding makes, with the Python-level field writes and address
 * lookups (several microseconds per step on the host cores) done here in one call.  No step
 * arithmetic happens here.
 *
 *   bind(rx_step_run_address)
 *   run(args_addr, io_addr, batch, tokens, tok_indptr, n_new, q, k_new, v_new, out, lse, d_stage,
 *       d_stage_bytes) -> rc
 *
 * tokens / tok_indptr / n_new: C-contiguous host arrays (int32 / int64 / int32; checked by the
 * caller), read through the buffer protocol; q, k_new, v_new, out, lse (or None): objects with
 * a data_ptr() method (device tensors); d_stage, d_stage_bytes: the device staging copy that goes
 * with this step's staging buffer (int address and size).  The GIL is released during the
 * native call. */
#define PY_SSIZE_T_CLEAN
#include <Python.h>

#include "radix_attn.h"

typedef int (*run_fn)(const rx_step_args*);
static run_fn g_run = NULL;
static PyObject* g_data_ptr = NULL;   /* interned "data_ptr" */

static int host_addr(PyObject* o, const void** out) {
    Py_buffer v;
    if (PyObject_GetBuffer(o, &v, PyBUF_SIMPLE) != 0) return -1;
    *out = v.buf;
    PyBuffer_Release(&v);   /* the caller holds the array for the whole call */
    return 0;
}

static int dev_addr(PyObject* o, void** out) {
    if (o == Py_None) {
        *out = NULL;
        return 0;
    }
    PyObject* r = PyObject_CallMethodNoArgs(o, g_data_ptr);
    if (!r) return -1;
    *out = PyLong_AsVoidPtr(r);
    Py_DECREF(r);
    return PyErr_Occurred() ? -1 : 0;
}

static PyObject* py_bind(PyObject* self, PyObject* arg) {
    (void)self;
    void* f = PyLong_AsVoidPtr(arg);
    if (PyErr_Occurred()) return NULL;
    if (!f) {
        PyErr_SetString(PyExc_ValueError, "bind: null function address");
        return NULL;
    }
    g_run = (run_fn)f;
    Py_RETURN_NONE;
}

static PyObject* py_run(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    (void)self;
    if (n != 13) {
        PyErr_SetString(PyExc_TypeError, "run: 13 arguments expected");
        return NULL;
    }
    if (!g_run) {
        PyErr_SetString(PyExc_RuntimeError, "run: bind() was not called");
        return NULL;
    }
    rx_step_args* args = (rx_step_args*)PyLong_AsVoidPtr(a[0]);
    rx_step_io* io = (rx_step_io*)PyLong_AsVoidPtr(a[1]);
    const long batch = PyLong_AsLong(a[2]);
    void* d_stage = PyLong_AsVoidPtr(a[11]);
    const size_t d_stage_bytes = PyLong_AsSize_t(a[12]);
    if (PyErr_Occurred()) return NULL;
    if (!args || !io || batch < 0 || batch > INT32_MAX) {
        PyErr_SetString(PyExc_ValueError, "run: bad struct address or batch");
        return NULL;
    }
    const void *tokens, *tok_indptr, *n_new;
    void *q, *k, *v, *out, *lse;
    if (host_addr(a[3], &tokens) || host_addr(a[4], &tok_indptr) || host_addr(a[5], &n_new) || dev_addr(a[6], &q) ||
        dev_addr(a[7], &k) || dev_addr(a[8], &v) || dev_addr(a[9], &out) || dev_addr(a[10], &lse))
        return NULL;
    io->d_q = q;
    io->d_k_new = k;
    io->d_v_new = v;
    io->d_out = out;
    io->d_lse = (float*)lse;
    io->d_stage = d_stage;
    io->d_stage_bytes = d_stage_bytes;
    args->batch = (int32_t)batch;
    args->tokens = (const int32_t*)tokens;
    args->tok_indptr = (const int64_t*)tok_indptr;
    args->n_new = (const int32_t*)n_new;
    int rc;
    Py_BEGIN_ALLOW_THREADS
    rc = g_run(args);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(rc);
}

static PyMethodDef methods[] = {
    {"bind", (PyCFunction)py_bind, METH_O, "bind(address of rx_step_run)"},
    {"run", (PyCFunction)(void (*)(void))py_run, METH_FASTCALL,
     "run(args_addr, io_addr, batch, tokens, tok_indptr, n_new, q, k_new, v_new, out, lse, d_stage, d_stage_bytes) -> rc"},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_rxstep", NULL, -1, methods, NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__rxstep(void) {
    g_data_ptr = PyUnicode_InternFromString("data_ptr");
    if (!g_data_ptr) return NULL;
    return PyModule_Create(&module);
}
