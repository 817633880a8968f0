"""The README's Python snippets stay in step with the package: each parses,
and every `zp.` / `zd.` name they use exists (CPU only; the snippets run on
a GPU and, for the exchanges, on several ranks)."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def snippets():
    text = open(os.path.join(ROOT, "README.md")).read()
    return re.findall(r"```python\n(.*?)```", text, re.S)


def test_readme_snippets_name_real_calls():
    import zero_partitioned_mixed_layout_gb300 as zp
    from zero_partitioned_mixed_layout_gb300 import dist as zd
    blocks = snippets()
    assert len(blocks) >= 3
    used = set()
    for code in blocks:
        tree = ast.parse(code)
        for node in ast.walk(tree):
            if isinstance(node, ast.Attribute) and isinstance(node.value, ast.Name) and node.value.id in ("zp", "zd"):
                used.add((node.value.id, node.attr))
    mods = {"zp": zp, "zd": zd}
    missing = [f"{m}.{a}" for m, a in sorted(used) if not hasattr(mods[m], a)]
    assert not missing, missing
    assert ("zd", "onebit_exchange_worker_signs") in used and ("zp", "zero_step") in used
