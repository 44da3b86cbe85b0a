"""The C-ABI library builds, loads without a GPU, and exports every declared symbol."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(gptk?_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from decoder_only_transformer_gpt_gb300 import build, binding
    build.build()
    return binding.load()


def test_headers_declare_the_boundary():
    names = declared_functions()
    for required in ("gpt_create", "gpt_forward", "gpt_destroy", "gpt_strerror", "gpt_forward_host",
                     "gpt_status", "gptk_gemm", "gptk_attention", "gptk_lmhead_ce"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_strerror_and_param_count(lib):
    from decoder_only_transformer_gpt_gb300 import binding
    from workloads import workload
    assert lib.gpt_strerror(0) == b"ok"
    assert b"T > ctx" in lib.gpt_strerror(binding.GPT_ESEQ)
    for name in ("toy", "minigpt", "gpt2_small", "gpt1_postnorm"):
        import oracle
        cfg = workload(name).cfg
        assert binding.param_count(cfg) == oracle.param_count(cfg)


def test_create_rejects_bad_config_without_gpu(lib):
    import ctypes
    from decoder_only_transformer_gpt_gb300 import binding
    from workloads import GPTConfig
    bad = binding.make_config(GPTConfig(V=17, C=16, H=3, L=1, ctx=12, ffn=64), 24)
    h = ctypes.c_void_p()
    assert lib.gpt_create(ctypes.byref(bad), None, ctypes.byref(h)) == binding.GPT_ECONFIG
    odd = binding.make_config(GPTConfig(V=17, C=12, H=2, L=1, ctx=12, ffn=64), 24)
    assert lib.gpt_create(ctypes.byref(odd), None, ctypes.byref(h)) == binding.GPT_EINVAL
    assert not h.value


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "decoder_only_transformer_gpt_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.replace("oracle-free", ""), f


def test_gradient_parameter_ids_match_the_binding():
    # gpt_grad's parameter ids (include/gpt.h) and the binding's names, in the same order
    from decoder_only_transformer_gpt_gb300 import binding
    text = open(os.path.join(ROOT, "include", "gpt.h")).read()
    ids = {k.lower(): int(v) for k, v in re.findall(r"\bGPT_P_(\w+)\s*=\s*(\d+)", text)}
    assert sorted(ids.values()) == list(range(len(binding.GRAD_PARAMS)))
    for i, name in enumerate(binding.GRAD_PARAMS):
        assert ids[name] == i, name


def test_gemm_pair_validates_arguments_before_the_device(lib):
    # every argument check of gptk_gemm_pair runs on the host before any device call (the pointers
    # below are never dereferenced); without a GPU the entry then reports GPT_ECONFIG (clusters of two
    # cannot be resident), never a launch
    import ctypes
    from decoder_only_transformer_gpt_gb300 import binding
    P = ctypes.c_void_p(0x10000)
    f = lib.gptk_gemm_pair
    resid, store = binding.EPI_BIAS_RESID, binding.EPI_F32
    assert f(None, P, None, P, 1, 8, 8, resid, 0, None) == binding.GPT_EINVAL          # no A
    assert f(P, P, None, P, 1, 8, 8, 7, 0, None) == binding.GPT_EINVAL                 # no such epilogue
    assert f(P, P, None, P, 1, 8, 64, store, 2, None) == binding.GPT_EINVAL            # split-K of a store
    assert f(P, P, P, P, 1, 8, 64, resid, 2, None) == binding.GPT_EINVAL               # split-K with a bias
    assert f(P, P, None, P, 1, 8, 64, resid, 2, None) == binding.GPT_EINVAL            # 2 slices of 1 K block
    assert f(P, P, None, P, 1, 8, 12, resid, 0, None) == binding.GPT_EINVAL            # K not a multiple of 8
    assert f(P, P, None, P, 0, 8, 8, resid, 0, None) == binding.GPT_OK                 # nothing to do
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert f(P, P, None, P, 1, 8, 8, resid, 0, None) == binding.GPT_ECONFIG
