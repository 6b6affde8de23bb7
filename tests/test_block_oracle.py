"""The scheduler / block-manager oracle against its pins, and planted mistakes against the pins
(no GPU). A mutant is a text edit of a temporary copy of ``oracle/block_manager.py``."""
import importlib.util
import sys

import pytest

import pins_blocks
from oracle import block_manager

SOURCE = block_manager.__file__


@pytest.mark.parametrize("pin", pins_blocks.ALL_PINS, ids=[p.__name__ for p in pins_blocks.ALL_PINS])
def test_oracle_pin(pin):
    pin(block_manager)


# (name, original text, planted text)
MUTANTS = [
    ("free_list_lifo", "b = self.free.popleft()\n        self.ref[b] = 1",
     "b = self.free.pop()\n        self.ref[b] = 1"),
    ("oldest_victim", "victim = max(self.running, key=lambda x: x.arrival)",
     "victim = min(self.running, key=lambda x: x.arrival)"),
    ("no_copy_on_write", "if self.ref[last] > 1:", "if False:"),
    ("cow_keeps_reference", "self.ref[last] -= 1", "pass"),
    ("prompt_not_shared", "self.ref[b] = len(g.seqs)", "self.ref[b] = 1"),
    ("growth_ignores_sharing", "return 1 if self.ref[s.table[-1]] > 1 else 0", "return 0"),
    ("swap_out_leaks", "for _ in range(refs):\n                        self._release(b)",
     "self._release(b)"),
    ("swap_in_reversed", "s.table = [to_gpu[c] for c in s.table]",
     "s.table = [to_gpu[c] for c in reversed(s.table)]"),
    ("recompute_drops_pending", "total = s.length + 1", "total = s.length"),
    ("retire_late", "s.generated >= g.max_new_tokens", "s.generated > g.max_new_tokens"),
    ("append_slot_off_by_one", "writes.append((s, s.length, b * self.B + s.length % self.B))",
     "writes.append((s, s.length, b * self.B + (s.length + 1) % self.B))"),
    ("waiting_back_of_queue", "self.waiting.appendleft(victim)", "self.waiting.append(victim)"),
    ("oversized_group_accepted", "if not 1 <= num_samples <= min(256, self.max_running):",
     "if not 1 <= num_samples <= 256:"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not found; update the mutant"
    path = tmp_path / f"bm_{name}.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"bm_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod  # dataclasses look their module up while the class is built
    try:
        spec.loader.exec_module(mod)
    finally:
        del sys.modules[spec.name]
    caught = []
    for pin in pins_blocks.ALL_PINS:
        try:
            pin(mod)
        except Exception as exc:  # AssertionError, or an error from inconsistent bookkeeping
            caught.append(f"{pin.__name__}: {type(exc).__name__}")
    assert caught, f"mutant {name} survived every pin"
