"""The C ABI library loads and exports every function include/pp.h declares; host-side
configuration checks (no GPU needed)."""
import ctypes
import os
import re

import pytest

import full_duplex_speech_lockstep_gb300 as pp
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "pp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pp_[a-z_]+)\s*\(", text)))


def test_every_declared_function_is_exported():
    lib = pp.lib()
    declared = _declared()
    assert declared == sorted(pp.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_weight_enum_matches_header():
    text = open(os.path.join(ROOT, "include", "pp.h")).read()
    names = re.findall(r"\bPP_W_([A-Z_]+)\s*[,=]", text)
    names = [n.lower() for n in names if n != "COUNT"]
    # header name -> binding name: matrices carry a "w" prefix in the binding
    rename = {"qkv": "wqkv", "o": "wo", "gu": "wgu", "down": "wdown", "text": "wtext",
              "dep_qkv": "dep_wqkv", "dep_o": "dep_wo", "dep_gu": "dep_wgu",
              "dep_down": "dep_wdown"}
    assert [rename.get(n, n) for n in names] == pp.WEIGHT_NAMES
    assert pp.WEIGHT_NAMES == synth.weight_names()


def test_weight_shapes_match_generator():
    for shape in [synth.TINY, synth.SMALL, synth.FULL]:
        cfg = pp.make_config(shape, 4)
        specs = {n: (shp, dt) for n, shp, dt, _ in synth.weight_specs(shape)}
        for i, name in enumerate(pp.WEIGHT_NAMES):
            dims, f32 = pp.pp_weight_shape(cfg, i)
            assert dims == specs[name][0], name
            assert f32 == (specs[name][1] == "f32"), name


def test_workspace_size_and_config_validation():
    full = pp.pp_workspace_bytes(pp.make_config(synth.FULL, 64))
    ring = 32 * 64 * 2 * 32 * 3000 * 128 * 2
    assert ring <= full < ring + (1 << 30)
    assert pp.pp_workspace_bytes(pp.make_config(synth.FULL, 1)) < full
    bad = pp.make_config(synth.TINY, 0)
    with pytest.raises(pp.PPError):
        pp.pp_workspace_bytes(bad)
    bad = pp.make_config(synth.TINY, 65)
    with pytest.raises(pp.PPError):
        pp.pp_workspace_bytes(bad)
    import dataclasses
    bad = pp.make_config(dataclasses.replace(synth.TINY, n_heads=3), 1)
    with pytest.raises(pp.PPError):
        pp.pp_workspace_bytes(bad)
    with pytest.raises(pp.PPError):
        pp.pp_weight_shape(pp.make_config(synth.TINY, 1), pp.PP_W_COUNT)


def test_create_rejects_bad_arguments_without_touching_the_gpu():
    cfg = pp.make_config(synth.TINY, 1)
    lib = pp.lib()
    h = ctypes.c_void_p()
    w = pp.pp_weights()
    # null weights / workspace are rejected before any CUDA call
    assert lib.pp_create(ctypes.byref(cfg), ctypes.byref(w), None, 0, ctypes.byref(h)) == pp.PP_EINVAL
    assert lib.pp_session_open(None, 0) == pp.PP_EINVAL
    assert lib.pp_step(None, None, None, None, None, None, None, None) == pp.PP_EINVAL


def test_sampling_rejects_bad_arguments_without_touching_the_gpu():
    lib = pp.lib()
    S = pp.sampling(text_temperature=0.7, text_top_p=0.9, seed=3)
    assert lib.pp_session_sampling(None, 0, ctypes.byref(S)) == pp.PP_EINVAL
    # rows == 0 is a no-op; every malformed argument is refused before any CUDA call
    ok = dict(ld=64, rows=0, n=64, T=0.7, k=0, p=0.9, R=1.0)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.pp_sample(None, a["ld"], a["rows"], a["n"], a["T"], a["k"], a["p"], a["R"],
                             None, 0, None, None, None, None, None)
    assert call() == pp.PP_OK
    assert call(rows=1) == pp.PP_EINVAL                 # null logits / uniforms / tokens
    assert call(n=0) == pp.PP_EINVAL
    assert call(ld=32) == pp.PP_EINVAL                  # n > ld
    assert call(n=60000, ld=60000) == pp.PP_EINVAL      # a row larger than shared memory
    assert call(T=0.0) == pp.PP_EINVAL
    assert call(T=float("nan")) == pp.PP_EINVAL
    assert call(p=0.0) == pp.PP_EINVAL
    assert call(p=1.5) == pp.PP_EINVAL
    assert call(R=0.0) == pp.PP_EINVAL
    assert lib.pp_sample(None, 64, 0, 64, 0.7, 0, 0.9, 1.0, ctypes.c_void_p(16), 300, None,
                         None, None, None, None) == pp.PP_EINVAL   # history without counts


def test_binding_structs_match_the_header_layout(tmp_path):
    """The ctypes structures mirror pp.h field for field: offsets and sizes from a C
    program compiled against the header equal the binding's."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    structs = {"pp_config": pp.pp_config, "pp_sampling": pp.pp_sampling,
               "pp_prompt": pp.pp_prompt, "pp_weights": pp.pp_weights}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "pp.h"', 'int main(void) {']
    for name, cls in structs.items():
        lines.append('  printf("%s size %%zu\\n", sizeof(%s));' % (name, name))
        for f in cls._fields_:
            lines.append('  printf("%s %s %%zu\\n", offsetof(%s, %s));' % (name, f[0], name, f[0]))
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.check_call(["gcc", "-std=c11", "-I", inc, str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for name, cls in structs.items():
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for f in cls._fields_:
            assert got[(name, f[0])] == getattr(cls, f[0]).offset, (name, f[0])


def test_fault_test_word_rejects_bad_arguments():
    """pp_test_faults validates on the host (a null engine, negative counts, unknown
    kernel families) before it touches the device."""
    lib = pp.lib()
    assert lib.pp_test_faults(None, 0, 0, 0, None) == pp.PP_EINVAL


def test_depformer_head_count_limit():
    """The depformer step attention takes one warp per head in one CTA: at most 16 heads,
    8 with head dim 128."""
    import dataclasses
    for dd, heads, good in [(1024, 16, True), (2048, 32, False), (1024, 8, True),
                            (2048, 16, False), (4096, 32, False), (512, 16, True)]:
        s = dataclasses.replace(synth.TINY, dep_d=dd, dep_heads=heads, dep_ffn=2 * dd)
        cfg = pp.make_config(s, 4)
        if good:
            assert pp.pp_workspace_bytes(cfg) > 0, (dd, heads)
        else:
            with pytest.raises(pp.PPError):
                pp.pp_workspace_bytes(cfg)


def test_low_latency_config_limits():
    """The persistent depformer serves engines of at most 8 slots on the tensor-core path."""
    ok = pp.make_config(synth.TINY, 8, pp.PP_FLAG_LOW_LATENCY)
    assert pp.pp_workspace_bytes(ok) > 0
    for cfg in [pp.make_config(synth.TINY, 9, pp.PP_FLAG_LOW_LATENCY),
                pp.make_config(synth.TINY, 4, pp.PP_FLAG_LOW_LATENCY | pp.PP_FLAG_CUDA_CORE_GEMM)]:
        with pytest.raises(pp.PPError):
            pp.pp_workspace_bytes(cfg)
