"""Host-only checks of the build helpers."""

import os
import shutil

from causal_linear_attention_la_gb300 import build as b


def test_kernel_digest_is_location_independent(monkeypatch, tmp_path):
    """The digest that keys the committed ncu traffic figures must not depend
    on where the tree is checked out (the GPU machine builds a copy elsewhere)."""
    names = ["la_decode.cu", "la_internal.cuh"]
    d0 = b.kernel_digest(names)
    root2 = tmp_path / "elsewhere"
    shutil.copytree(b.CSRC, root2 / "causal_linear_attention_la_gb300" / "csrc")
    shutil.copytree(b.INCLUDE, root2 / "include")
    pkg2 = str(root2 / "causal_linear_attention_la_gb300")
    moved = {b.INCLUDE: str(root2 / "include"), b.CSRC: os.path.join(pkg2, "csrc")}
    monkeypatch.setattr(b, "NVCC_FLAGS", [moved.get(f, f) for f in b.NVCC_FLAGS])
    monkeypatch.setattr(b, "ROOT", str(root2))
    monkeypatch.setattr(b, "PKG", pkg2)
    monkeypatch.setattr(b, "CSRC", os.path.join(pkg2, "csrc"))
    monkeypatch.setattr(b, "INCLUDE", str(root2 / "include"))
    assert b.kernel_digest(names) == d0
    # and it does change with the sources
    with open(os.path.join(pkg2, "csrc", "la_decode.cu"), "a") as f:
        f.write("\n// changed\n")
    assert b.kernel_digest(names) != d0
