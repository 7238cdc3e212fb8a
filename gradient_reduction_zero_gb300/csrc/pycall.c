/* CPython entry points for the compute calls of libdpz.so (include/dpz.h).
 *
 * Each function takes the C call's arguments as Python ints in the same order
 * (device addresses, sizes, dtype codes, the address of a dpz_adamw_cfg, the
 * stream handle; None for a NULL pointer), converts each once and makes the
 * call.  It returns the call's status code.  Nothing else happens here: the
 * checks, the error message and the launches are the library's.  The point is
 * the cost of a call from Python, which for the launch-bound workloads is most
 * of a step: a vectorcall with a fixed argument list instead of ctypes'
 * per-argument conversion objects.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>

#include <limits.h>
#include <stdint.h>
#include <string.h>

#include "dpz.h"

typedef union {
    void* p;
    int64_t l;
    int i;
} Arg;

/* fmt: one character per argument, 'p' pointer (int or None), 'l' int64,
 * 'i' int.  Sets a Python exception and returns -1 on a bad argument. */
static int parse(PyObject* const* a, Py_ssize_t n, const char* fmt, Arg* out)
{
    const Py_ssize_t k = (Py_ssize_t)strlen(fmt);
    if (n != k) {
        PyErr_Format(PyExc_TypeError, "expected %zd arguments, got %zd", k, n);
        return -1;
    }
    for (Py_ssize_t j = 0; j < k; ++j) {
        PyObject* o = a[j];
        if (fmt[j] == 'p') {
            if (o == Py_None) {
                out[j].p = NULL;
                continue;
            }
            out[j].p = PyLong_AsVoidPtr(o);
            if (out[j].p == NULL && PyErr_Occurred()) return -1;
        } else if (fmt[j] == 'l') {
            const long long v = PyLong_AsLongLong(o);
            if (v == -1 && PyErr_Occurred()) return -1;
            out[j].l = (int64_t)v;
        } else {
            const long v = PyLong_AsLong(o);
            if (v == -1 && PyErr_Occurred()) return -1;
            if (v < INT_MIN || v > INT_MAX) {
                PyErr_SetString(PyExc_OverflowError, "argument does not fit a C int");
                return -1;
            }
            out[j].i = (int)v;
        }
    }
    return 0;
}

#define CALL(name, fmt, nargs, expr)                                             \
    static PyObject* py_##name(PyObject* self, PyObject* const* a, Py_ssize_t n) \
    {                                                                            \
        (void)self;                                                              \
        Arg s[nargs];                                                            \
        if (parse(a, n, fmt, s)) return NULL;                                    \
        return PyLong_FromLong((long)(expr));                                    \
    }

#define F(k) ((float*)s[k].p)
#define CFG(k) ((const dpz_adamw_cfg*)s[k].p)

CALL(dp_reduce_scatter_avg, "pliip", 5, dp_reduce_scatter_avg(s[0].p, s[1].l, s[2].i, s[3].i, s[4].p))
CALL(dp_allreduce_avg, "pliip", 5, dp_allreduce_avg(s[0].p, s[1].l, s[2].i, s[3].i, s[4].p))
CALL(dp_grad_global_norm, "pliippp", 7,
     dp_grad_global_norm(s[0].p, s[1].l, s[2].i, s[3].i, s[4].p, F(5), s[6].p))
CALL(dp_grad_global_norm_static, "pliipp", 6,
     dp_grad_global_norm_static(s[0].p, s[1].l, s[2].i, s[3].i, F(4), s[5].p))
CALL(zero1_adamw_step, "pppppliiippp", 12,
     zero1_adamw_step(s[0].p, F(1), F(2), F(3), s[4].p, s[5].l, s[6].i, s[7].i, s[8].i, CFG(9),
                      s[10].p, s[11].p))
CALL(dp_allgather, "pliip", 5, dp_allgather(s[0].p, s[1].l, s[2].i, s[3].i, s[4].p))
CALL(dp_zero1_step, "pppppliiipppp", 13,
     dp_zero1_step(s[0].p, F(1), F(2), F(3), s[4].p, s[5].l, s[6].i, s[7].i, s[8].i, CFG(9),
                   s[10].p, F(11), s[12].p))
CALL(dp_reduce_scatter_avg_range, "pliillpip", 9,
     dp_reduce_scatter_avg_range(s[0].p, s[1].l, s[2].i, s[3].i, s[4].l, s[5].l, s[6].p, s[7].i,
                                 s[8].p))
CALL(dp_reduce_scatter_avg_bucket, "pllpliipip", 10,
     dp_reduce_scatter_avg_bucket(s[0].p, s[1].l, s[2].l, s[3].p, s[4].l, s[5].i, s[6].i, s[7].p,
                                  s[8].i, s[9].p))
CALL(dp_grad_norm_finalize, "plipp", 5, dp_grad_norm_finalize(s[0].p, s[1].l, s[2].i, F(3), s[4].p))
CALL(dp_zero1_update, "pppppliiippp", 12,
     dp_zero1_update(s[0].p, F(1), F(2), F(3), s[4].p, s[5].l, s[6].i, s[7].i, s[8].i, CFG(9),
                     s[10].p, s[11].p))
CALL(dp_zero2_update, "pppppliiippp", 12,
     dp_zero2_update(s[0].p, F(1), F(2), F(3), s[4].p, s[5].l, s[6].i, s[7].i, s[8].i, CFG(9),
                     s[10].p, s[11].p))

#define ENTRY(name) {#name, (PyCFunction)(void (*)(void))py_##name, METH_FASTCALL, NULL}

static PyMethodDef methods[] = {
    ENTRY(dp_reduce_scatter_avg),
    ENTRY(dp_allreduce_avg),
    ENTRY(dp_grad_global_norm),
    ENTRY(dp_grad_global_norm_static),
    ENTRY(zero1_adamw_step),
    ENTRY(dp_allgather),
    ENTRY(dp_zero1_step),
    ENTRY(dp_reduce_scatter_avg_range),
    ENTRY(dp_reduce_scatter_avg_bucket),
    ENTRY(dp_grad_norm_finalize),
    ENTRY(dp_zero1_update),
    ENTRY(dp_zero2_update),
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {
    PyModuleDef_HEAD_INIT, "_dpzcall",
    "The compute calls of libdpz.so, with Python ints for arguments.", -1, methods,
    NULL, NULL, NULL, NULL,
};

PyMODINIT_FUNC PyInit__dpzcall(void) { return PyModule_Create(&module); }
