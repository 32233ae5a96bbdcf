"""The Python binding's view of the C ABI matches include/mlora.h: the ctypes structures have the
C structures' field offsets and sizes (a small C program built with the host compiler prints
them), and every prototype's argument count and integer widths match the binding's table."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

import adapter_gemv_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mlora.h")


def c_layout(tmp_path, struct, fields):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    src = tmp_path / "layout.c"
    lines = [f'printf("%s %zu %zu\\n", "{f}", offsetof({struct}, {f}), sizeof((({struct} *)0)->{f}));'
             for f in fields]
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "mlora.h"\nint main(void) {\n'
                   + "\n".join(lines) + f'\nprintf("sizeof %zu 0\\n", sizeof({struct}));\nreturn 0;\n}}\n')
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", f"-I{os.path.dirname(HEADER)}", str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    return {name: (int(a), int(b)) for name, a, b in (ln.split() for ln in out if ln)}


@pytest.mark.parametrize("struct, cls", [("mlora_pool", m.mlora_pool), ("mlora_problem", m.mlora_problem),
                                         ("mlora_group", m.mlora_group)])
def test_struct_layouts_match(tmp_path, struct, cls):
    names = [f for f, _ in cls._fields_]
    c = c_layout(tmp_path, struct, names)
    for f, _ in cls._fields_:
        desc = getattr(cls, f)
        assert (desc.offset, desc.size) == c[f], f"{struct}.{f}: ctypes {(desc.offset, desc.size)} vs C {c[f]}"
    assert ctypes.sizeof(cls) == c["sizeof"][0]


def prototypes():
    src = open(HEADER).read()
    out = {}
    for name, args in re.findall(r"MLORA_API\s+int\s+(lora_\w+)\s*\(([^)]*)\)", src):
        out[name] = [a.strip() for a in args.split(",") if a.strip() and a.strip() != "void"]
    return out


def width(c_arg: str):
    """'p' for any pointer, else the integer width in bits."""
    if "*" in c_arg:
        return "p"
    for t, w in (("int64_t", 64), ("int32_t", 32), ("uint32_t", 32), ("uint64_t", 64), ("int ", 32), ("size_t", 64)):
        if c_arg.startswith(t):
            return w
    raise AssertionError(f"unhandled C argument type: {c_arg}")


def ctypes_width(t):
    if t in (ctypes.c_void_p,) or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "p"
    return 8 * ctypes.sizeof(t)


def test_prototypes_match_the_binding_table():
    protos = prototypes()
    for name, sig in m.SIGNATURES.items():
        assert name in protos, f"{name} is not declared in mlora.h"
        c_args = protos[name]
        assert len(c_args) == len(sig), f"{name}: {len(c_args)} C arguments, {len(sig)} in the binding"
        for i, (ca, pt) in enumerate(zip(c_args, sig)):
            assert width(ca) == ctypes_width(pt), f"{name} argument {i} ({ca}) vs {pt}"
    # every int-returning entry point that takes arguments is in the table
    missing = [n for n, a in protos.items() if a and n not in m.SIGNATURES and n != "lora_set_programmatic_launch"]
    assert not missing, f"not in the binding's table: {missing}"
