"""The C-ABI library on a host without a GPU: it loads, exports every
symbol the header declares, and rejects bad arguments on the host before
touching a device."""
import ctypes
import os
import re

import pytest
import torch

from block_fp8_mixture_route_gb300 import _lib, api, synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_fp8_block.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return _lib.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_fp8_block_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    assert sorted(names) == sorted(_lib.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_strings(lib):
    assert lib.moe_fp8_block_abi_version() == _lib.ABI_VERSION
    for code in [0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -10, 12345]:
        assert len(_lib.error_string(code)) > 0
    assert lib.moe_fp8_block_last_path() == _lib.MOE_PATH_NONE


def _descs(prob):
    return [api.desc(prob[n]) for n in ("hidden", "topk_ids", "topk_weights", "w13", "w13_scale", "w2", "w2_scale")]


def _call(lib, prob, out=None, s13=None, s2=None, opt=None, mutate=None):
    d = _descs(prob)
    o = api.desc(out if out is not None else torch.empty(prob["hidden"].shape, dtype=torch.bfloat16))
    if mutate:
        mutate(d, o)
    s13 = prob["w13_scale"].stride(1) if s13 is None else s13
    s2 = prob["w2_scale"].stride(1) if s2 is None else s2
    P = ctypes.byref
    if opt is None:
        return lib.moe_fp8_block_forward(P(d[0]), P(d[1]), P(d[2]), P(d[3]), P(d[4]), s13, P(d[5]), P(d[6]), s2,
                                         P(o), None)
    return lib.moe_fp8_block_forward_ex(P(d[0]), P(d[1]), P(d[2]), P(d[3]), P(d[4]), s13, P(d[5]), P(d[6]), s2,
                                        P(o), None, P(opt))


@pytest.fixture(scope="module")
def tiny():
    return syn.make_problem(syn.TINY, T=4, seed=0)


def test_null_descriptor(lib):
    P = ctypes.byref
    t = api.desc(torch.zeros(4, 256, dtype=torch.bfloat16))
    assert lib.moe_fp8_block_forward(None, P(t), P(t), P(t), P(t), 2, P(t), P(t), 1, P(t), None) == -1


@pytest.mark.parametrize("case,code", [
    ("hidden_dtype", -2), ("ids_dtype", -2), ("w13_dtype", -2),
    ("H_not_128", -3), ("out_shape", -3), ("scale_rows", -3),
    ("s13_small", -5), ("s2_mismatch", -5), ("w13_noncontig", -5),
    ("unaligned_hidden", -4), ("alias", -6), ("k_zero", -3), ("null_data", -1),
])
def test_argument_errors(lib, tiny, case, code):
    prob = dict(tiny)
    out = None
    s13 = s2 = None
    mutate = None
    if case == "hidden_dtype":
        prob["hidden"] = tiny["hidden"].float()
    elif case == "ids_dtype":
        prob["topk_ids"] = tiny["topk_ids"].long() if False else tiny["topk_ids"].float()
    elif case == "w13_dtype":
        prob["w13"] = tiny["w13"].to(torch.int32)
    elif case == "H_not_128":
        def mutate(d, o):
            d[0].shape[1] = 200
            o.shape[1] = 200
    elif case == "out_shape":
        out = torch.empty(3, 256, dtype=torch.bfloat16)
    elif case == "scale_rows":
        prob["w2_scale"] = tiny["w2_scale"][:, :1]
    elif case == "s13_small":
        s13 = 1
    elif case == "s2_mismatch":
        s2 = 3
    elif case == "w13_noncontig":
        prob["w13"] = tiny["w13"].transpose(1, 2)
    elif case == "unaligned_hidden":
        big = torch.zeros(4 * 256 + 8, dtype=torch.bfloat16)
        prob["hidden"] = big[1:1 + 4 * 256].view(4, 256)
    elif case == "alias":
        out = tiny["hidden"]
    elif case == "k_zero":
        prob["topk_ids"] = tiny["topk_ids"][:, :0]
        prob["topk_weights"] = tiny["topk_weights"][:, :0]
    elif case == "null_data":
        def mutate(d, o):
            d[3].data = None
    if case == "k_zero":
        rc = _call(lib, prob, out, s13, s2, mutate=mutate)
        assert rc in (-3, -9)
        return
    assert _call(lib, prob, out, s13, s2, mutate=mutate) == code


def test_bad_options(lib, tiny):
    o = _lib.MoeOptions()
    o.force_path = 7
    assert _call(lib, tiny, opt=o) == -9
    o = _lib.MoeOptions()
    o.reserved[1] = 1
    assert _call(lib, tiny, opt=o) == -9
    o = _lib.MoeOptions()
    o.decode_act = 2              # neither MOE_DECODE_ACT_BF16 nor _E4M3
    assert _call(lib, tiny, opt=o) == -9
    for field, bad in (("decode_kernel", 2), ("decode_kernel", -1), ("debug_wait_timeout_us", -5),
                       ("debug_wait_timeout_us", 1000001), ("debug_drop_stage", -1)):
        o = _lib.MoeOptions()
        setattr(o, field, bad)
        assert _call(lib, tiny, opt=o) == -9, (field, bad)


def test_empty_batch_is_noop(lib):
    prob = syn.make_problem(syn.TINY, T=0, seed=0)
    assert _call(lib, prob) == 0


def test_no_device_is_reported(lib, tiny):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = _call(lib, tiny)
    assert rc in (-8, -10)
    assert lib.moe_fp8_block_route(ctypes.byref(api.desc(tiny["topk_ids"])), 8, 1, 1, 1, 1, 1, 1, None) in (-8, -10)


def test_route_argument_errors(lib, tiny):
    d = api.desc(tiny["topk_ids"])
    P = ctypes.byref
    assert lib.moe_fp8_block_route(P(d), 0, 1, 1, 1, 1, 1, 1, None) == -9
    assert lib.moe_fp8_block_route(P(d), 8, None, 1, 1, 1, 1, 1, None) == -1
    f = api.desc(tiny["topk_weights"])
    assert lib.moe_fp8_block_route(P(f), 8, 1, 1, 1, 1, 1, 1, None) == -2


def test_act_quant_argument_errors(lib):
    P = ctypes.byref
    x = api.desc(torch.zeros(2, 200, dtype=torch.bfloat16))
    assert lib.moe_fp8_block_act_quant(P(x), 16, 16, None) == -3
    x = api.desc(torch.zeros(2, 256, dtype=torch.float32))
    assert lib.moe_fp8_block_act_quant(P(x), 16, 16, None) == -2


def test_reserve_argument_errors(lib):
    assert lib.moe_fp8_block_reserve(16, 0, 2048, 512, 128, None) == -9
    assert lib.moe_fp8_block_reserve(16, 8, 2000, 512, 128, None) == -9


def _call_bias(lib, prob, b13, b2, out=None):
    d = _descs(prob)
    o = api.desc(out if out is not None else torch.empty(prob["hidden"].shape, dtype=torch.bfloat16))
    P = ctypes.byref
    db13 = api.desc(b13) if b13 is not None else None
    db2 = api.desc(b2) if b2 is not None else None
    return lib.moe_fp8_block_forward_bias(P(d[0]), P(d[1]), P(d[2]), P(d[3]), P(d[4]), prob["w13_scale"].stride(1),
                                          P(d[5]), P(d[6]), prob["w2_scale"].stride(1),
                                          P(db13) if db13 is not None else None,
                                          P(db2) if db2 is not None else None, P(o), None, None)


def test_bias_argument_errors(lib, tiny):
    E, H, I = syn.TINY.E, syn.TINY.H, syn.TINY.I
    b13, b2 = syn.make_biases(syn.TINY)
    if not torch.cuda.is_available():
        # valid arguments get as far as the device check (host tensors: never
        # make this call where a GPU could run it)
        assert _call_bias(lib, tiny, b13, b2) in (-8, -10)
        assert _call_bias(lib, tiny, None, None) in (-8, -10)
    assert _call_bias(lib, tiny, b13.to(torch.bfloat16), b2) == -2         # fp32 only
    assert _call_bias(lib, tiny, b13[:, :I], b2) == -3                     # [E, 2I]
    assert _call_bias(lib, tiny, b13, b2[:E - 1]) == -3                    # [E, H]
    assert _call_bias(lib, tiny, b13.t().contiguous().t(), b2) == -5       # stride[1] != 1
    wide = torch.zeros(E, 2 * I + 2)
    assert _call_bias(lib, tiny, wide[:, :2 * I], b2) == -5                # expert stride not a multiple of 4
    big = torch.zeros(E * H + 1)
    assert _call_bias(lib, tiny, b13, big[1:].view(E, H)) == -4            # 16-byte alignment
    alias = torch.zeros(E * H, dtype=torch.float32)
    assert _call_bias(lib, tiny, b13, alias.view(E, H), out=alias.view(torch.bfloat16)[:4 * H].view(4, H)) == -6


@pytest.mark.parametrize("H,I,ok", [(192, 144, True), (320, 176, True), (2880, 2880, True), (160, 256, False),
                                    (256, 136, False), (64, 256, False), (256, 112, False)])
def test_ragged_shape_rules(lib, H, I, ok):
    """H must be a multiple of 64 and I of 16, both at least 128; multiples
    of 128 are not required (ragged layers run on the prefill path)."""
    shp = syn.MoeShape(E=2, H=H, I=I, k=2)
    prob = syn.make_problem(shp, T=1, seed=0)
    if ok and torch.cuda.is_available():
        pytest.skip("host tensors: the valid call is only made without a GPU")
    rc = _call(lib, prob)
    if ok:
        assert rc in (-8, -10)          # past every argument check, then no device
    else:
        assert rc == -3


@pytest.mark.parametrize("T,k,E,H,I,path", [
    (16, 8, 128, 2048, 512, 1),    # small layer: decode up to T*k = E
    (17, 8, 128, 2048, 512, 2),
    (1, 8, 256, 2560, 640, 1),     # 4-row-pair decode units: decode only up to 8 slots
    (2, 8, 256, 2560, 640, 2),
    (8, 8, 256, 2560, 640, 2),
    (1, 8, 256, 7168, 2048, 2),    # 3 decode ring stages: always the grouped GEMMs
    (1, 4, 16, 320, 192, 1),       # ragged, multiples of 64: decode
    (1, 4, 16, 320, 176, 2),       # I not a multiple of 64: prefill only
    (0, 8, 128, 2048, 512, 1),
])
def test_default_path_rule(lib, T, k, E, H, I, path):
    """The default gate as a host-only query: decode while T*k <= E, the
    decode gate/up ring keeps at least 4 stages and its units are whole
    8-row-pair blocks (H <= 2048) or the batch routes at most 8 slots."""
    assert lib.moe_fp8_block_default_path(T, k, E, H, I) == path
    assert api.moe_fp8_block_default_path(T, k, E, H, I) == path


def test_default_path_argument_errors(lib):
    err_arg, err_shape = -9, -3   # MOE_ERR_ARG, MOE_ERR_SHAPE
    assert lib.moe_fp8_block_default_path(-1, 8, 128, 2048, 512) == err_arg
    assert lib.moe_fp8_block_default_path(1, 0, 128, 2048, 512) == err_arg
    assert lib.moe_fp8_block_default_path(1, 8, 0, 2048, 512) == err_arg
    assert lib.moe_fp8_block_default_path(1, 8, 128, 160, 512) == err_shape
    with pytest.raises(RuntimeError):
        api.moe_fp8_block_default_path(1, 8, 128, 160, 512)


C_CHECK = r"""
#include "moe_fp8_block.h"
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#define CHECK(c) do { if (!(c)) { printf("failed: %s\n", #c); return 1; } } while (0)

int main(void) {
  static const int codes[] = {MOE_OK, MOE_ERR_NULL, MOE_ERR_DTYPE, MOE_ERR_SHAPE, MOE_ERR_ALIGN, MOE_ERR_STRIDE,
                              MOE_ERR_ALIAS, MOE_ERR_CAPTURE_GROW, MOE_ERR_CUDA, MOE_ERR_ARG, MOE_ERR_DEVICE};
  static uint16_t host[4 * 256];
  moe_tensor t;
  size_t i;
  CHECK(moe_fp8_block_abi_version() == MOE_FP8_BLOCK_ABI_VERSION);
  for (i = 0; i < sizeof(codes) / sizeof(codes[0]); ++i) {
    const char* s = moe_fp8_block_error_string(codes[i]);
    CHECK(s != NULL && strlen(s) > 0);
  }
  CHECK(moe_fp8_block_default_path(1, 8, 128, 2048, 512) == MOE_PATH_DECODE);
  CHECK(moe_fp8_block_default_path(1, 8, 256, 7168, 2048) == MOE_PATH_PREFILL);
  CHECK(moe_fp8_block_default_path(-1, 8, 128, 2048, 512) == MOE_ERR_ARG);
  memset(&t, 0, sizeof(t));
  t.data = host;
  t.ndim = 2;
  t.dtype = MOE_BF16;
  t.shape[0] = 4;
  t.shape[1] = 256;
  t.stride[0] = 256;
  t.stride[1] = 1;
  CHECK(moe_fp8_block_forward(NULL, &t, &t, &t, &t, 2, &t, &t, 1, &t, NULL) == MOE_ERR_NULL);
  CHECK(moe_fp8_block_last_path() == MOE_PATH_NONE);
  moe_fp8_block_release();
  printf("ok\n");
  printf("moe_tensor %u data %u ndim %u dtype %u shape %u stride %u\n", (unsigned)sizeof(moe_tensor),
         (unsigned)offsetof(moe_tensor, data), (unsigned)offsetof(moe_tensor, ndim),
         (unsigned)offsetof(moe_tensor, dtype), (unsigned)offsetof(moe_tensor, shape),
         (unsigned)offsetof(moe_tensor, stride));
  printf("moe_options %u gate_ratio %u force_path %u decode_act %u decode_kernel %u debug_wait_timeout_us %u "
         "debug_drop_stage %u reserved %u\n", (unsigned)sizeof(moe_options),
         (unsigned)offsetof(moe_options, gate_ratio), (unsigned)offsetof(moe_options, force_path),
         (unsigned)offsetof(moe_options, decode_act), (unsigned)offsetof(moe_options, decode_kernel),
         (unsigned)offsetof(moe_options, debug_wait_timeout_us), (unsigned)offsetof(moe_options, debug_drop_stage),
         (unsigned)offsetof(moe_options, reserved));
  return 0;
}
"""


def test_header_is_plain_c(lib):
    """The header compiles as strict C99 (and as C++), and a C program links
    the library and calls it without Python: the boundary is a C ABI."""
    import shutil
    import subprocess
    from block_fp8_mixture_route_gb300 import build
    gcc, gxx = shutil.which("gcc"), shutil.which("g++")
    if not gcc:
        pytest.skip("no C compiler")
    out_dir = os.path.join(build.BUILD, "abi_c_check")
    os.makedirs(out_dir, exist_ok=True)
    src, exe = os.path.join(out_dir, "check.c"), os.path.join(out_dir, "check")
    with open(src, "w") as f:
        f.write(C_CHECK)
    libdir = os.path.dirname(_lib.LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.dirname(HEADER), src,
                    "-L", libdir, "-lmoe_fp8_block", "-Wl,-rpath," + libdir, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    lines = r.stdout.strip().splitlines()
    assert r.returncode == 0 and lines and lines[0] == "ok", r.stdout + r.stderr
    # the binding's structures have the layout a C compiler gives the header's
    for line, cls in zip(lines[1:], (_lib.MoeTensor, _lib.MoeOptions)):
        f = line.split()
        assert int(f[1]) == ctypes.sizeof(cls), line
        layout = {f[i]: int(f[i + 1]) for i in range(2, len(f), 2)}
        assert layout == {name: getattr(cls, name).offset for name, _ in cls._fields_}, line
    if gxx:
        subprocess.run([gxx, "-std=c++11", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-x", "c++",
                        "-I", os.path.dirname(HEADER), src], check=True)


def _header_signatures():
    """{function: (return type, [parameter types])} from the header's text."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    sigs = {}
    for ret, name, params in re.findall(r"((?:const\s+)?\w+\s*\*?)\s*(moe_fp8_block_\w+)\s*\(([^)]*)\)\s*;", src):
        types = []
        for prm in params.split(","):
            prm = " ".join(prm.split())
            if prm in ("", "void"):
                continue
            types.append(re.sub(r"\s*\b\w+$", "", prm).replace(" *", "*"))
        sigs[name] = (" ".join(ret.split()).replace(" *", "*"), types)
    return sigs


def test_binding_signatures_match_header(lib):
    """Every ctypes argtype/restype of the binding is the C type the header
    declares (a mismatched width would pass garbage through the ABI)."""
    P = ctypes.POINTER
    vp = ctypes.c_void_p
    ctype = {
        "const moe_tensor*": P(_lib.MoeTensor), "moe_tensor*": P(_lib.MoeTensor),
        "const moe_options*": P(_lib.MoeOptions),
        "int64_t": ctypes.c_int64, "int32_t": ctypes.c_int32, "int": ctypes.c_int,
        "uint32_t*": P(ctypes.c_uint32), "void* const*": P(ctypes.c_void_p),
        "void*": vp, "const void*": vp, "uint8_t*": vp, "const uint8_t*": vp, "float*": vp, "int32_t*": vp,
    }
    rtype = {"int": ctypes.c_int, "const char*": ctypes.c_char_p, "void": None}
    sigs = _header_signatures()
    assert sorted(sigs) == sorted(_lib.EXPORTS)
    for name, (ret, params) in sigs.items():
        fn = getattr(lib, name)
        assert fn.restype == rtype[ret], name
        assert len(fn.argtypes) == len(params), name
        for i, (have, want) in enumerate(zip(fn.argtypes, params)):
            assert have == ctype[want], f"{name} argument {i}: {want}"
